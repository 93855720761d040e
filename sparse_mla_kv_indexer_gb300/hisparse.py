"""ctypes binding of libhisparse.so, the C ABI declared in include/hisparse.h.

Argument marshalling only: every computation runs in the library's CUDA
kernels. Tensors are passed by ``data_ptr()`` and the stream is torch's current
stream unless one is given. Importing this module loads the library and raises
ImportError when it has not been built, so nothing can silently fall back.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libhisparse.so")

STATUS = {
    0: "HS_OK", 1: "HS_ERR_INVALID", 2: "HS_ERR_OOM", 3: "HS_ERR_CAPACITY", 4: "HS_ERR_CUDA",
    5: "HS_ERR_TIMEOUT", 6: "HS_ERR_HOST_MISSING", 7: "HS_ERR_BAD_ID", 8: "HS_ERR_BAD_WEIGHT",
    9: "HS_ERR_SCRATCH_LIMIT", 10: "HS_ERR_NOT_RESOLVED", 11: "HS_ERR_RANGE",
}
SELECT_AUTO, SELECT_LOCAL = 0, 1   # HS_SELECT_AUTO, HS_SELECT_LOCAL
PLAN_PAD, PLAN_RESIDENT, PLAN_HIT, PLAN_MISS = 0, 1, 2, 3
IDX_INT8, IDX_FP8 = 0, 1       # HS_IDX_INT8, HS_IDX_FP8
IDX_FP8_PAGE_BYTES = 8448      # 64 x 128 e4m3 key bytes, then 64 fp32 scales
MAX_CTX = 1310720            # HS_MAX_CTX: longest context a pool accepts


class HisparseError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call}: {STATUS.get(status, status)}")
        self.status = status


class PoolConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "page_size", "row_bytes", "idx_dim", "n_idx_heads", "n_heads", "topk", "n_layers",
        "layers_per_indexer", "num_pages", "num_idx_pages", "max_requests", "max_ctx",
        "max_q_per_req", "hot_rows", "max_tokens", "idx_format")] + [("host_pages", ctypes.c_int64)]


class PlanEntry(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("slot", ctypes.c_int32), ("row", ctypes.c_int32),
                ("evicted", ctypes.c_int32)]


class Counters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("resident", "hits", "misses", "h2d_bytes", "d2h_bytes")] + \
               [("reserved", ctypes.c_uint64 * 3)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIGS = {
    "hs_pool_config_check": [ctypes.POINTER(PoolConfig)],
    "hs_pool_init": [ctypes.POINTER(PoolConfig), ctypes.POINTER(_P), ctypes.POINTER(_P), _P, ctypes.POINTER(_P)],
    "hs_pool_destroy": [_P],
    "hs_request_set_pages": [_P, _I, _I, _I, _P, _P, _P, _P],
    "hs_hot_lease": [_P, _I, _I, _I, _P, _P],
    "hs_hot_release": [_P, _I, _P],
    "hs_append_rows": [_P, _I, _P, _P, _P, _P, _P],
    "hs_indexer_topk": [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P],
    "hs_indexer_topk_noalloc": [_P, _I, _I, _P, _P, _P, _P, _P, _P],
    "hs_indexer_topk_fp8": [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P],
    "hs_resolve_topk": [_P, _I, _I, _I, _P, _P, _P, _P, _P],
    "hs_replay_topk": [_P, _I, _I, _P, _P, _P, _P],
    "hs_sparse_mla_decode": [_P, _I, _I, _P, _P, ctypes.c_float, _P, _P, _P],
    "hs_offload_pages": [_P, _I, _P, _P, _P],
    "hs_get_error": [_P, ctypes.POINTER(ctypes.c_int), _P],
    "hs_set_select_mode": [_P, _I],
    "hs_select_selftest": [_P, _I, _P, _P, _P],
    "hs_get_counters": [_P, ctypes.POINTER(Counters), _I, _P],
    "hs_link_probe": [_P, ctypes.c_int64, _I, _P, ctypes.c_int64, _P, _P],
    "hs_wait_selftest": [_P, _P],
}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.hs_status_string.argtypes = [ctypes.c_int]
    lib.hs_status_string.restype = ctypes.c_char_p
    return lib


lib = _load()


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name: str, st: int) -> None:
    if st != 0:
        raise HisparseError(name, st)


def _host_array(values, ctype):
    if values is None:
        return None
    arr = (ctype * len(values))(*[int(v) for v in values])
    return ctypes.cast(arr, _P), arr


def config_ok(cfg: PoolConfig) -> bool:
    """hs_pool_config_check: whether hs_pool_init would accept this geometry (no GPU needed)."""
    return lib.hs_pool_config_check(ctypes.byref(cfg)) == 0


def link_probe(host_rows, row_bytes: int, src_rows, dst, stream=None) -> None:
    """hs_link_probe: copy dst[i] = host row src_rows[i] (single-row reads from a
    pinned, mapped host tensor), the access pattern of the resolver's miss copies."""
    _check("hs_link_probe", lib.hs_link_probe(_ptr(host_rows), host_rows.numel() * host_rows.element_size() // row_bytes,
                                              row_bytes, _ptr(src_rows), src_rows.numel(), _ptr(dst), _stream(stream)))


class Pool:
    """A HiSparse pool over caller-owned KV tensors, index caches and a pinned host pool."""

    def __init__(self, cfg: PoolConfig, kv_layers: Sequence, idx_layers: Sequence, host_kv):
        self.cfg = cfg
        self._keep = (list(kv_layers), list(idx_layers), host_kv)
        kv = (_P * len(kv_layers))(*[_ptr(t) for t in kv_layers])
        ix = (_P * len(idx_layers))(*[_ptr(t) for t in idx_layers])
        handle = _P()
        _check("hs_pool_init", lib.hs_pool_init(ctypes.byref(cfg), kv, ix, _ptr(host_kv), ctypes.byref(handle)))
        self.handle = handle

    def close(self) -> None:
        if self.handle:
            _check("hs_pool_destroy", lib.hs_pool_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- host-side residency updates ------------------------------------------------
    def set_pages(self, req: int, first_page: int, block_table=None, idx_pages=None, host_pages=None,
                  stream=None) -> None:
        n = len(next(x for x in (block_table, idx_pages, host_pages) if x is not None))
        bt = _host_array(block_table, ctypes.c_int32)
        ip = _host_array(idx_pages, ctypes.c_int32)
        hp = _host_array(host_pages, ctypes.c_int64)
        _check("hs_request_set_pages", lib.hs_request_set_pages(
            self.handle, req, first_page, n, bt and bt[0], ip and ip[0], hp and hp[0], _stream(stream)))

    def hot_lease(self, req: int, group: int, pages, stream=None) -> None:
        arr = _host_array(pages, ctypes.c_int32)
        _check("hs_hot_lease", lib.hs_hot_lease(self.handle, req, group, len(pages), arr[0], _stream(stream)))

    def hot_release(self, req: int, stream=None) -> None:
        _check("hs_hot_release", lib.hs_hot_release(self.handle, req, _stream(stream)))

    # -- device hot path -------------------------------------------------------------
    def append_rows(self, req, pos, kv_rows, idx_keys, stream=None) -> None:
        _check("hs_append_rows", lib.hs_append_rows(self.handle, req.numel(), _ptr(req), _ptr(pos), _ptr(kv_rows),
                                                    _ptr(idx_keys), _stream(stream)))

    def indexer_topk(self, index_layer: int, req, limit, q, w, topk, scores=None, stream=None) -> None:
        _check("hs_indexer_topk", lib.hs_indexer_topk(self.handle, index_layer, req.numel(), _ptr(req), _ptr(limit),
                                                      _ptr(q), _ptr(w), _ptr(topk), _ptr(scores), _stream(stream)))

    def indexer_topk_fp8(self, index_layer: int, req, limit, q, w, topk, scores=None, stream=None) -> None:
        """FP8 keys (pool idx_format IDX_FP8): q e4m3 bytes, w fp32, scores nullable fp32."""
        _check("hs_indexer_topk_fp8", lib.hs_indexer_topk_fp8(self.handle, index_layer, req.numel(), _ptr(req),
                                                              _ptr(limit), _ptr(q), _ptr(w), _ptr(topk), _ptr(scores),
                                                              _stream(stream)))

    def indexer_topk_noalloc(self, index_layer: int, req, limit, q, w, topk, stream=None) -> None:
        """hs_indexer_topk with its score scratch in the library's fixed array, for
        callers that cannot allocate device memory (see include/hisparse.h)."""
        _check("hs_indexer_topk_noalloc", lib.hs_indexer_topk_noalloc(
            self.handle, index_layer, req.numel(), _ptr(req), _ptr(limit), _ptr(q), _ptr(w), _ptr(topk),
            _stream(stream)))

    def resolve_topk(self, group: int, step: int, req, topk, row_ids, plan=None, stream=None) -> None:
        _check("hs_resolve_topk", lib.hs_resolve_topk(self.handle, group, step, req.numel(), _ptr(req), _ptr(topk),
                                                      _ptr(row_ids), _ptr(plan), _stream(stream)))

    def replay_topk(self, group: int, req, topk, row_ids, stream=None) -> None:
        """Row ids of an already resolved selection, without touching the LRU state."""
        _check("hs_replay_topk", lib.hs_replay_topk(self.handle, group, req.numel(), _ptr(req), _ptr(topk),
                                                    _ptr(row_ids), _stream(stream)))

    def sparse_mla_decode(self, layer: int, q, row_ids, sm_scale: float, out, lse=None, stream=None) -> None:
        _check("hs_sparse_mla_decode", lib.hs_sparse_mla_decode(self.handle, layer, q.shape[0], _ptr(q),
                                                                _ptr(row_ids), float(sm_scale), _ptr(out),
                                                                _ptr(lse), _stream(stream)))

    def offload_pages(self, pool_pages, host_pages, stream=None) -> None:
        _check("hs_offload_pages", lib.hs_offload_pages(self.handle, pool_pages.numel(), _ptr(pool_pages),
                                                        _ptr(host_pages), _stream(stream)))

    # -- status --------------------------------------------------------------------
    def get_error(self, stream=None) -> int:
        v = ctypes.c_int(0)
        _check("hs_get_error", lib.hs_get_error(self.handle, ctypes.byref(v), _stream(stream)))
        return v.value

    def set_select_mode(self, mode: int) -> None:
        """hs_set_select_mode: SELECT_LOCAL keeps the top-K selection off grid-wide waits."""
        _check("hs_set_select_mode", lib.hs_set_select_mode(self.handle, mode))

    def select_selftest(self, limit, topk, stream=None) -> None:
        """hs_select_selftest: the grid-wide selection with one CTA per token withholding
        its arrivals, so the others time out (HS_ERR_TIMEOUT, half-used scratch)."""
        _check("hs_select_selftest", lib.hs_select_selftest(self.handle, limit.numel(), _ptr(limit), _ptr(topk),
                                                            _stream(stream)))

    def wait_selftest(self, stream=None) -> None:
        """hs_wait_selftest: a bounded device wait that runs out (HS_ERR_TIMEOUT)."""
        _check("hs_wait_selftest", lib.hs_wait_selftest(self.handle, _stream(stream)))

    def raise_on_device_error(self, stream=None) -> None:
        st = self.get_error(stream)
        if st:
            raise HisparseError("device", st)

    def counters(self, reset: bool = False, stream=None) -> Counters:
        c = Counters()
        _check("hs_get_counters", lib.hs_get_counters(self.handle, ctypes.byref(c), int(reset), _stream(stream)))
        return c
