"""The multi-rank path of bench.py on CPU, with world size 2 over gloo.

bench.py runs one rank per GPU under torch.distributed.run: each rank times an
independent copy of the workload (its own seed; the path needs no exchange),
the ranks meet at a barrier on both sides of the timed region, and rank 0
reports the maximum time over ranks.  These tests exercise that logic without
a GPU: the helpers through two spawned gloo ranks, and the oracle arm
(``--impl reference``, which needs no GPU) end to end under torch.distributed.run.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    from exact_tiled_attention_08_gb300.workloads import WORKLOADS

    r, wsz, local = bench.dist_setup()
    assert (r, wsz, local) == (rank, world, rank)
    bench.barrier(wsz)
    # max over ranks of a per-rank time
    m = bench.max_over_ranks(1.5 + rank, wsz)
    # each rank draws its own copy of the workload
    inp, _ = bench.cpu_inputs(WORKLOADS["tiny_b1_h1_n128_d128"], seed_offset=7919 * rank)
    gathered = [torch.zeros_like(inp["q"].float()) for _ in range(wsz)]
    import torch.distributed as dist

    dist.all_gather(gathered, inp["q"].float())
    bench.barrier(wsz)
    dist.destroy_process_group()
    out.put((rank, m, bool(torch.equal(gathered[0], gathered[1]))))


@pytest.mark.skipif(torch.cuda.is_available(), reason="gloo CPU ranks; the GPU box runs the NCCL path")
def test_rank_helpers_world_size_2():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(2))
    assert [r for r, _, _ in res] == [0, 1]
    assert all(m == 2.5 for _, m, _ in res)          # the maximum over ranks, on every rank
    assert all(not same for _, _, same in res)        # independent inputs per rank


def test_reference_arm_under_torchrun_world_size_2():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny_b1_h1_n128_d128", "--steps", "2", "--warmup", "1",
           "--gpus", "2"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(x) for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
