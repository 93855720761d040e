"""The number of library kernels one decode step launches, as bench.py reports it.

One step of the bench session (device-resident inputs, so the step issues
nothing but library calls) is captured into a CUDA graph through the CUDA
runtime; its kernel nodes are counted, and every node whose function the
runtime names must be a kernel of the library (namespace ``hs``). The count
must equal ``BenchSession.launches``.
"""
import ctypes

import pytest

from sparse_mla_kv_indexer_gb300 import schedule as S
from sparse_mla_kv_indexer_gb300 import workload as W

pytestmark = pytest.mark.gpu


class _KernelNodeParams(ctypes.Structure):
    _fields_ = [("func", ctypes.c_void_p), ("grid", ctypes.c_uint * 3), ("block", ctypes.c_uint * 3),
                ("shared_mem", ctypes.c_uint), ("kernel_params", ctypes.c_void_p), ("extra", ctypes.c_void_p)]


def _graph_kernels(rt, graph):
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * n.value)()
    assert rt.cudaGraphGetNodes(graph, nodes, ctypes.byref(n)) == 0
    names = []
    for node in nodes:
        kind = ctypes.c_int(-1)
        assert rt.cudaGraphNodeGetType(ctypes.c_void_p(node), ctypes.byref(kind)) == 0
        if kind.value != 0:   # cudaGraphNodeTypeKernel
            continue
        # the function's name where the runtime reports it (nodes made by extended
        # launches may not expose it); the count is what the bench claims
        p = _KernelNodeParams()
        name = ctypes.c_char_p()
        if (rt.cudaGraphKernelNodeGetParams(ctypes.c_void_p(node), ctypes.byref(p)) == 0
                and rt.cudaFuncGetName(ctypes.byref(name), ctypes.c_void_p(p.func)) == 0 and name.value):
            names.append(name.value.decode())
        else:
            rt.cudaGetLastError()
            names.append(None)
    return names


@pytest.mark.parametrize("name", ["tiny", "small_groups", "small_batch"])
def test_step_kernel_count_matches_bench_claim(name):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_indexer_gb300.driver import BenchSession, GpuRun
    rt = ctypes.CDLL("libcudart.so.13")   # the runtime torch has loaded
    cfg = W.named_config(name)
    wl = W.Workload(cfg)
    sch = S.Schedule(cfg)
    plans = [sch.plan(s) for s in range(cfg.steps)]
    run = GpuRun(wl, sch.setup)
    stream = torch.cuda.Stream()
    try:
        with torch.cuda.stream(stream):
            sess = BenchSession(run, plans, mode="device")
            sess.tick(0)
            sess.step(0)     # the first calls set kernel attributes; later steps are only captured
            stream.synchronize()
            run.pool.raise_on_device_error(stream)
            checked = 0
            for i in range(1, cfg.steps):
                sess.tick(i)
                stream.synchronize()
                graph = ctypes.c_void_p()
                assert rt.cudaStreamBeginCapture(ctypes.c_void_p(stream.cuda_stream), 0) == 0
                sess.step(i)
                assert rt.cudaStreamEndCapture(ctypes.c_void_p(stream.cuda_stream), ctypes.byref(graph)) == 0
                try:
                    names = _graph_kernels(rt, graph)
                finally:
                    rt.cudaGraphDestroy(graph)
                assert names and all(n is None or n.startswith("_ZN2hs") or "hs::" in n for n in names), names
                assert len(names) == sess.launches(i), (i, names)
                checked += 1
            assert checked == cfg.steps - 1
    finally:
        run.close()
