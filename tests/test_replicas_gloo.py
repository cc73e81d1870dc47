"""The N > 1 bench path on CPU with the gloo backend, world size 2.

`bench.py --gpus N` runs N independent replicas (the layer has no cross-GPU
step here): the timed region's length is the slowest rank's, and `value` is
all ranks' tokens over that time.  These tests check that host logic without
a GPU: the max-over-ranks reduction in two gloo processes, and a torchrun
launch of the reference arm, where rank 0 alone prints its line.
"""

import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.5 + rank, world, "cpu")
        out[rank] = (ms, bench.replica_value(4096, world, 20, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_value_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5                  # both ranks see the slowest rank's time
    assert res[0][1] == res[1][1] == 2 * 4096 * 20 / 2.5e-3


def test_reference_arm_under_torchrun_prints_one_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "tiny_fp8"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    # the rest of the line's contract: the metric and unit of the arm it is
    # compared with, the workload it sampled, and a CPU baseline that is the
    # line's own value
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["steps"] == 1 and d["warmup"] == 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "tiny_fp8" and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["value"] == d["value"] and cb["unit"] == "tokens/s" and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
