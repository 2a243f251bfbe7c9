"""Host logic of bench.py, on the CPU: the counted work, the ncu traffic
lookup, the multi-rank helpers over a world-size-2 gloo group, and the
reference arm's rank handling and JSON line."""
from __future__ import annotations

import importlib.util
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("T,causal,W", [(1, True, 0), (7, True, 0), (64, True, 0), (50, True, 8), (50, True, 1),
                                        (50, True, 50), (33, False, 0), (40, False, 7), (40, False, 60)])
def test_visible_pairs_match_brute_force(T, causal, W):
    b = _bench()
    w = b.WORKLOADS[3].replace(T=T, causal=causal, window=W)
    i, j = np.arange(T)[:, None], np.arange(T)[None, :]
    vis = np.ones((T, T), bool)
    if causal:
        vis &= j <= i
    if W:
        vis &= (i - j) < W
    want = float(vis.sum())
    if causal and not W or (causal and W >= T):
        want = T * T / 2.0  # the metric counts the causal triangle as half the square
    assert b.visible_pairs(w) == want


def test_counted_work_of_the_windowed_workload():
    b = _bench()
    w = b.WORKLOADS[4]
    pairs = w.T * w.window - w.window * (w.window - 1) // 2  # 7,864,832 per head
    assert pairs == 7864832 and b.visible_pairs(w) == pairs
    f = b.counted_flops(w)
    assert f["fwd"] == 4 * w.B * w.H * w.D * pairs and f["fwd_bwd"] == 10 * w.B * w.H * w.D * pairs
    work = b.kernel_work(w, 2)
    assert work["fwd"][1] + work["bwd_dkdv"][1] + work["bwd_dq"][1] == 18 * w.B * w.H * w.D * pairs
    assert work["bwd_preprocess"] == ("hbm", 2.0 * w.B * w.H * w.T * w.D * 2 + 4.0 * w.B * w.H * w.T)


def test_traffic_lookup_needs_matching_source_hash(tmp_path):
    b = _bench()
    name = b.WORKLOADS[5].name
    lines = open(os.path.join(ROOT, "profiles", "ncu_traffic.txt")).read()
    for kernel in ("fwd", "bwd_dkdv", "bwd_dq"):
        if f"kernel={kernel};" in lines and f"sha={b.source_sha(b.KERNEL_SOURCES[kernel])};" in lines:
            assert b.ncu_traffic(kernel, name) > 0
    assert b.ncu_traffic("bwd_dkdv", "no such workload") is None
    b.source_sha = lambda _: "0000000000000000"
    assert b.ncu_traffic("bwd_dkdv", name) is None  # a changed kernel invalidates its counters


_RANK_SCRIPT = r"""
import os, sys, json
import torch.distributed as dist
sys.path.insert(0, {root!r})
import importlib.util
spec = importlib.util.spec_from_file_location("bench_rank", os.path.join({root!r}, "bench.py"))
b = importlib.util.module_from_spec(spec); spec.loader.exec_module(b)
dist.init_process_group("gloo", init_method="env://")
rank, world = dist.get_rank(), dist.get_world_size()
b.barrier(world)
m = b.max_over_ranks(1.5 + 2.0 * rank, world)
b.barrier(world)
print(json.dumps({{"rank": rank, "max": m}}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_and_barrier_on_two_gloo_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                   LOCAL_RANK=str(rank))
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK_SCRIPT.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["max"] == 3.5 for o in outs)  # max over ranks of 1.5 + 2 * rank


def _run_reference(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "1", "--ref-T", "256", "--workload", "3"], env=env, capture_output=True,
                          text=True, timeout=300)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _run_reference(1)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_reference(0)
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"] and line["higher_is_better"] is True
