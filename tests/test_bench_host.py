"""Host-side checks of bench.py: multi-rank aggregation over gloo (world size 2, CPU) and the
JSON line of the reference arm's helpers that need no GPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took (r + 1) seconds and did (r + 1) * 10 units
    t, u = bench.aggregate(float(rank + 1), float((rank + 1) * 10), world)
    q.put((rank, t, u))
    dist.destroy_process_group()


def test_aggregate_max_time_sum_units_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, u in res:
        assert t == 2.0 and u == 30.0


def test_single_rank_aggregate_is_identity():
    import bench
    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)


def test_visible_pairs_union_matches_oracle_counts():
    """The bench's visible-pair count (union of each row's slots) on a CPU tensor table."""
    import numpy as np
    import torch

    import bench
    from masked_flashattention_gb300 import workloads as W
    from oracle import masks as M

    class FakeDesc:
        pass

    for wid in (1, 3, 4, 5):
        S = 1024
        seg, nseg = W.segments(wid, 2, S, seed=wid)
        tabs = np.stack([M.interval_table_fwd(wid, seg[b], int(nseg[b]), S) for b in range(2)])
        d = FakeDesc()
        d.ni_f = tabs.shape[1]
        d.itab_f = torch.from_numpy(tabs.reshape(-1).copy())
        got = bench.visible_pairs(d, 2, S)
        want = [int(M.dense_mask(wid, seg[b], int(nseg[b]), S).sum()) for b in range(2)]
        assert got == want


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` times the CPU oracle and prints one JSON line."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--config", "1", "--steps", "1", "--warmup", "3", "--ref-rows", "64"],
                         capture_output=True, text=True, timeout=300, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
