"""The committed DRAM-traffic table that bench.py reports as `roofline.traffic`.

Every entry comes from single-kernel ncu captures: one kernel (`-k`), one launch (`-c 1`),
clocks left alone (`--clock-control none`); its bytes are the sum over the call's kernels,
and it names the sources whose sha256 decides whether the bench may still use it.
"""
import json
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_mla_kv_indexer_gb300", "csrc")


def _table():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        return {k: v for k, v in json.load(f).items() if not k.startswith("_")}


def test_traffic_entries_come_from_single_kernel_captures():
    t = _table()
    assert t, "no entries"
    for key, ent in t.items():
        call, workload = key.split("@")
        assert call and workload
        assert ent["bytes_per_launch"] == sum(ent["kernels"].values()), key
        assert len(ent["commands"]) == len(ent["kernels"]), key
        for cmd, kernel in zip(ent["commands"], ent["kernels"]):
            assert "--clock-control none" in cmd, cmd
            assert re.search(r"(^|\s)-c 1(\s|$)", cmd), cmd
            m = re.search(r"-k regex:(\S+)", cmd)
            assert m and m.group(1) == kernel, (cmd, kernel)
            assert "|" not in m.group(1), cmd
            assert "bench.py" in cmd and f"--workload {workload}" in cmd, cmd
        for src in ent["sources"]:
            assert os.path.exists(os.path.join(CSRC, src)), src
        assert re.fullmatch(r"[0-9a-f]{64}", ent["source_sha256"]), key


def test_launch_lists_collect_only_the_duration():
    prof = os.path.join(ROOT, "profiles")
    names = [n for n in os.listdir(prof) if n.startswith("launches_")]
    assert names
    for n in names:
        text = open(os.path.join(prof, n)).read()
        for line in text.splitlines():
            if line.startswith("    ncu "):   # an indented command line
                assert "--metrics gpu__time_duration.sum " in line and "--clock-control none" in line, (n, line)
