"""The multi-process bench logic on CPU: two gloo ranks, barrier-bracketed
timing, slowest rank reported, work summed over ranks (replicas, weak
scaling).  No GPU; the per-rank step is a stand-in sleep."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    # rank-dependent timed total over 4 steps: rank 1 is slower
    total_ms = 40.0 * (rank + 1)
    ms, value = bench.aggregate(total_ms, 4, 1e12, 1e12, ws, "cpu")
    out[rank] = (ms, value)
    dist.destroy_process_group()


def test_two_rank_gloo_max_time_and_summed_work():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1]
    t, value = out[0]
    assert t == pytest.approx(20.0)          # the slowest rank: 80 ms / 4 steps
    assert value == pytest.approx(100.0)     # 2 ranks x 1 TFLOP per 20 ms step


def test_reference_arm_loads_no_library():
    """The reference arm (the fp64 oracle on the host cores) draws its inputs
    with `synth` on the host and takes lambda_init from the oracle: it runs
    without a GPU and never loads the CUDA library (checked in a fresh
    process, whose mapped files must not include it)."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import json, types, bench\n"
            "args = types.SimpleNamespace(workload='v1_fwd_f32', steps=2, warmup=1)\n"
            "bench.run_reference(args, 1, 0)\n"
            "from differential_attention_diff_gb300 import binding\n"
            "maps = open('/proc/self/maps').read()\n"
            "print(json.dumps({'lib': binding._lib is not None, 'mapped': 'libdiffattn' in maps}))\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                         timeout=300, check=True).stdout.strip().splitlines()
    line, probe = json.loads(out[-2]), json.loads(out[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["sample"]
    assert probe == {"lib": False, "mapped": False}
