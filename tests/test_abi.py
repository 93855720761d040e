"""The C-ABI library builds, loads and exports every symbol include/hisparse.h
declares; host-side argument checks answer HS_ERR_INVALID without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hisparse.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_mla_kv_indexer_gb300 import build
    path = build.LIB
    if not os.path.exists(path):
        build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hs_[a-z_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for want in ["hs_pool_init", "hs_pool_destroy", "hs_indexer_topk", "hs_resolve_topk",
                 "hs_sparse_mla_decode", "hs_offload_pages", "hs_get_error", "hs_append_rows",
                 "hs_request_set_pages", "hs_hot_lease", "hs_hot_release", "hs_get_counters",
                 "hs_status_string"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_status_strings(lib):
    lib.hs_status_string.restype = ctypes.c_char_p
    assert lib.hs_status_string(0) == b"ok"
    assert lib.hs_status_string(3) == b"hot buffer capacity exceeded"
    assert lib.hs_status_string(99) == b"unknown status"


def test_null_pool_is_invalid(lib):
    P = ctypes.c_void_p
    assert lib.hs_pool_destroy(None) == 1
    assert lib.hs_hot_release(None, 0, None) == 1
    assert lib.hs_indexer_topk(None, 0, 1, P(1), P(1), P(1), P(1), P(1), None, None) == 1
    assert lib.hs_resolve_topk(None, 0, 0, 1, P(1), P(1), P(1), None, None) == 1
    assert lib.hs_sparse_mla_decode(None, 0, 1, P(16), P(16), ctypes.c_float(1.0), P(16), None, None) == 1
    assert lib.hs_offload_pages(None, 1, P(1), P(1), None) == 1
    st = ctypes.c_int(0)
    assert lib.hs_get_error(None, ctypes.byref(st), None) == 1


def test_bad_geometry_is_invalid(lib):
    from sparse_mla_kv_indexer_gb300.hisparse import PoolConfig
    good = dict(page_size=64, row_bytes=656, idx_dim=128, n_idx_heads=64, n_heads=64, topk=2048,
                n_layers=4, layers_per_indexer=4, num_pages=100, num_idx_pages=100, max_requests=1,
                max_ctx=4096, max_q_per_req=1, hot_rows=4096, max_tokens=1, idx_format=0, host_pages=10)
    ptrs = (ctypes.c_void_p * 8)(*([16] * 8))
    out = ctypes.c_void_p()
    for key, bad in [("page_size", 32), ("row_bytes", 640), ("idx_dim", 64), ("n_heads", 48),
                     ("topk", 100), ("topk", 4096), ("max_ctx", 1000), ("hot_rows", 100),
                     ("max_q_per_req", 5), ("max_tokens", 0), ("n_idx_heads", 8), ("n_idx_heads", 24),
                     ("n_idx_heads", 80), ("hot_rows", 16384 + 64), ("num_pages", 1 << 25), ("num_idx_pages", 0),
                     ("host_pages", 0), ("max_ctx", 1310720 + 128), ("n_layers", 65), ("layers_per_indexer", 9),
                     ("idx_format", 2), ("max_tokens", 1025)]:
        cfg = PoolConfig(**{**good, key: bad})
        assert lib.hs_pool_config_check(ctypes.byref(cfg)) == 1, key
        assert lib.hs_pool_init(ctypes.byref(cfg), ptrs, ptrs, ctypes.c_void_p(16), ctypes.byref(out)) == 1, key
    for key, ok in [("n_idx_heads", 16), ("n_idx_heads", 48), ("n_heads", 16), ("topk", 128), ("max_q_per_req", 4),
                    ("hot_rows", 16384), ("max_ctx", 1310720), ("idx_format", 1), ("layers_per_indexer", 8)]:
        assert lib.hs_pool_config_check(ctypes.byref(PoolConfig(**{**good, key: ok}))) == 0, key
    assert lib.hs_pool_config_check(None) == 1
    cfg = PoolConfig(**good)
    assert lib.hs_pool_config_check(ctypes.byref(cfg)) == 0
    misaligned = (ctypes.c_void_p * 8)(*([24] * 8))
    assert lib.hs_pool_init(ctypes.byref(cfg), misaligned, ptrs, ctypes.c_void_p(16), ctypes.byref(out)) == 1


def test_binding_constants_match_the_header():
    from sparse_mla_kv_indexer_gb300 import hisparse as H
    text = open(HEADER).read()
    defines = dict(re.findall(r"#define\s+(HS_[A-Z_]+)\s+\(?([0-9a-fx]+(?:ll)?(?:\s*<<\s*\d+)?)\)?", text))
    assert int(defines["HS_MAX_CTX"]) == H.MAX_CTX
    assert H.MAX_CTX % 128 == 0 and H.MAX_CTX < (1 << 21)   # token ids fit the 21-bit tie-break field
    for code, name in H.STATUS.items():
        assert re.search(rf"\b{name}\s*=\s*{code}\b", text), name


@pytest.mark.parametrize("name", ["tiny", "ctx128k", "batch32", "ctx1m", "multiturn", "small_single", "small_batch",
                                  "small_groups", "small_reuse", "short_ctx", "tiny_fp8", "ctx128k_fp8", "ctx1m_fp8",
                                  "small_batch_fp8"])
def test_every_workload_geometry_is_accepted(lib, name):
    """The pool each workload builds passes hs_pool_config_check, so no shape fails
    only at hs_pool_init on the GPU."""
    from sparse_mla_kv_indexer_gb300 import schedule as S
    from sparse_mla_kv_indexer_gb300 import workload as W
    from sparse_mla_kv_indexer_gb300.driver import pool_config
    cfg = W.named_config(name)
    pc = pool_config(W.Workload(cfg), S.Schedule(cfg).setup)
    assert lib.hs_pool_config_check(ctypes.byref(pc)) == 0


def test_a_c_program_builds_and_calls_the_library(lib, tmp_path):
    """The header is plain C (C99, no C++ needed): a C program includes it, links
    libhisparse.so, and calls the host-only entry points."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from sparse_mla_kv_indexer_gb300 import build
    src = tmp_path / "abi_check.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "hisparse.h"
int main(void) {
  hs_pool_config c;
  memset(&c, 0, sizeof c);
  c.page_size = 64; c.row_bytes = 656; c.idx_dim = 128; c.n_idx_heads = 64; c.n_heads = 64;
  c.topk = 2048; c.n_layers = 4; c.layers_per_indexer = 4; c.num_pages = 100; c.num_idx_pages = 100;
  c.max_requests = 1; c.max_ctx = 131072; c.max_q_per_req = 1; c.hot_rows = 4096; c.max_tokens = 1;
  c.idx_format = HS_IDX_INT8; c.host_pages = 10;
  if (hs_pool_config_check(&c) != HS_OK) return 1;
  c.topk = 100;
  if (hs_pool_config_check(&c) != HS_ERR_INVALID) return 2;
  if (strcmp(hs_status_string(HS_ERR_CAPACITY), "hot buffer capacity exceeded") != 0) return 3;
  if (hs_sparse_mla_decode(NULL, 0, 1, NULL, NULL, 1.0f, NULL, NULL, NULL) != HS_ERR_INVALID) return 4;
  printf("ok\n");
  return 0;
}
''')
    exe = tmp_path / "abi_check"
    lib_dir = os.path.dirname(build.LIB)
    name = os.path.basename(build.LIB)[3:-3]          # libhisparse.so -> hisparse
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I" + os.path.join(ROOT, "include"), str(src),
                    "-L" + lib_dir, "-l" + name, "-Wl,-rpath," + lib_dir, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)
