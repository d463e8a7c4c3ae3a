"""Host-side logic of bench.py on the CPU: the whole-job aggregation across
ranks (two gloo processes), the useful-pair count, the reference arm's
JSON line (the fp64 oracle timed on a small sample), and the source keys of
the stored DRAM counts."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    dist = bench.Dist()
    # rank r processed (r+1)*10 units in (r+1) seconds
    value, slowest = bench.aggregate(10.0 * (rank + 1), 1.0 * (rank + 1), dist)
    dist.barrier()
    out[rank] = (value, slowest)
    dist.close()


def test_aggregate_over_two_gloo_ranks():
    world = 2
    port = 29500 + os.getpid() % 2000
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    # whole job: (10 + 20) units over the slowest rank's 2 s
    for r in range(world):
        assert res[r] == pytest.approx((15.0, 2.0))


def test_single_process_aggregate_is_identity():
    import bench
    d = bench.Dist()
    assert d.world == 1 or "WORLD_SIZE" in os.environ
    value, slowest = bench.aggregate(42.0, 2.0, d)
    assert (value, slowest) == (21.0, 2.0)


def test_useful_pairs_counts_visited_keys():
    import bench
    W = 4
    gate = np.array([[0, 1, 0, 0, 1, 0, 1]], np.uint8)
    # window rows: min(i+1, W); routed rows: i+1
    want = 1 + 2 + 3 + 4 + 5 + 4 + 7
    assert bench.useful_pairs(gate, W) == want


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3", "--ref-step-budget", "0.1"],
                         capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["steps"] == 1


def test_traffic_counts_resolve_for_the_current_sources():
    """Every stored DRAM count is keyed by the source text of its kernel (a
    whole file or a file up to a marker).  Each marker must still occur once
    in its file, and every kernel with a stored count has a source entry."""
    import bench
    csrc = os.path.join(ROOT, "sliding_window_attention_router_gb300", "csrc")
    for kernel, entries in bench.KERNEL_SOURCES.items():
        for entry in entries:
            name, marker = (entry, None) if isinstance(entry, str) else entry
            text = open(os.path.join(csrc, name)).read()
            if marker is not None:
                assert text.count(marker) == 1, (kernel, name, marker)
        assert len(bench.kernel_source_hash(kernel)) == 16
    assert {k for k, _ in bench.MEASURED_TRAFFIC} == set(bench.KERNEL_SOURCES)
