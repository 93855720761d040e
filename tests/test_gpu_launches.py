"""The number of library kernels one decode step launches, as bench.py reports it.

The step's kernels are counted from the CUDA activity trace of one step and
compared with ``BenchSession.launches``; every one must come from the library.
"""
import pytest

from sparse_mla_kv_indexer_gb300 import schedule as S
from sparse_mla_kv_indexer_gb300 import workload as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "small_groups"])
def test_step_kernel_count_matches_bench_claim(name):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from torch.profiler import ProfilerActivity, profile

    from sparse_mla_kv_indexer_gb300.driver import BenchSession, GpuRun
    cfg = W.named_config(name)
    wl = W.Workload(cfg)
    sch = S.Schedule(cfg)
    plans = [sch.plan(s) for s in range(cfg.steps)]
    run = GpuRun(wl, sch.setup)
    try:
        sess = BenchSession(run, plans, mode="device")
        sess.tick(0)
        sess.step(0)
        torch.cuda.synchronize()
        for i in range(1, cfg.steps):
            sess.tick(i)
            with profile(activities=[ProfilerActivity.CUDA]) as prof:
                sess.step(i)
                torch.cuda.synchronize()
            names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA
                     and "memcpy" not in e.name.lower() and "memset" not in e.name.lower()]
            ours = [n for n in names if "hs::" in n]
            assert len(ours) == len(names), names
            assert len(ours) == sess.launches(i), (i, sorted(ours))
        run.pool.raise_on_device_error()
    finally:
        run.close()
