"""The end-to-end path the bench times: inputs copied from one packed pinned host
buffer per step, the step, the outputs copied back. Its outputs must equal those of
the same steps run with device-resident inputs (two pools over the same workload,
driven alike; every kernel is deterministic), and the step must copy its inputs in
one host-to-device copy. Outputs come back either written by the attention straight
into pinned host memory or by one copy, both checked."""
import numpy as np
import pytest

from sparse_mla_kv_indexer_gb300 import schedule as S
from sparse_mla_kv_indexer_gb300 import workload as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,host_write_max", [("tiny", None), ("small_batch", None), ("small_batch", 0)])
def test_host_mode_steps_match_device_mode(name, host_write_max):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_indexer_gb300.driver import BenchSession, GpuRun
    cfg = W.named_config(name)
    steps = min(cfg.steps, 4)
    outs = {}
    for mode in ("device", "host"):
        wl = W.Workload(cfg)
        sch = S.Schedule(cfg)
        run = GpuRun(wl, sch.setup)
        if host_write_max is not None:   # 0: the outputs come back by one copy
            BenchSession.HOST_WRITE_MAX, saved = host_write_max, BenchSession.HOST_WRITE_MAX
        try:
            sess = BenchSession(run, [sch.plan(s) for s in range(steps)], mode=mode)
        finally:
            if host_write_max is not None:
                BenchSession.HOST_WRITE_MAX = saved
        got = []
        for i in range(steps):
            sess.tick(i)
            sess.step(i)
            torch.cuda.synchronize()
            run.pool.raise_on_device_error()
            got.append((sess.out_host if mode == "host" else sess.out.cpu()).numpy().copy())
        outs[mode] = got
        if mode == "host":
            _, host, _ = sess.steps[0]
            assert set(host) == {"_pack", "_dpack", "_bytes"} and host["_pack"].is_pinned()
    for i in range(steps):
        assert np.array_equal(outs["device"][i], outs["host"][i]), i
