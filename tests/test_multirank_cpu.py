"""The multi-replica host logic of bench.py on two CPU ranks (gloo).

With N > 1 every rank is an independent replica of the step on its own inputs;
the only collectives are the barrier and the max-reduction of the timing, and
the whole-job throughput counts every rank's steps against the slowest rank.
"""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from tree_speculative_decoding_bastion_gb300 import inputs as I
        wl = I.WORKLOADS["tiny_v1024_f32"]
        inp = I.make_step_inputs(wl, bench.replica_seed(rank, 0), with_attention=False)
        digest = torch.tensor([float(np.asarray(inp.logits, dtype=np.float64).sum())])
        all_d = [torch.zeros(1) for _ in range(world)]
        dist.all_gather(all_d, digest)
        ms = bench.max_over_ranks(10.0 + rank, world)      # this rank's fake timed region
        dist.barrier()
        q.put((rank, ms, [float(x.item()) for x in all_d], bench.job_throughput(world, 100, ms)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_reduce_the_slowest_time_and_draw_their_own_inputs():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, digests, value in res:
        assert ms == 11.0                          # both ranks hold the slowest rank's time
        assert digests[0] != digests[1]            # each replica drew its own batch
        assert value == pytest.approx(world * 100 / 0.011)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_v1024_f32", "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    import json
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_v1024_f32", "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_runs_the_steps_it_is_given():
    """The reference arm times exactly --steps steps after --warmup untimed
    ones (the counts in the line are the ones it ran), and reports the
    all-cores figure with its core count beside a one-core figure."""
    import json
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_v1024_f32", "--steps", "3", "--warmup", "2"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["steps"] == 3 and line["warmup"] == 2
    cpu = line["cpu_baseline"]
    assert cpu["cores"] >= 1 and cpu["one_core"]["cores"] == 1 and cpu["one_core"]["value"] > 0
    assert "model" in line["value_model"] and line["ms_per_step"] > 0
