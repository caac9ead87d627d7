"""The N > 1 path of bench.py is replicas (no collective on the data path):
its host-side aggregation -- the slowest rank's time, all ranks' units over
it -- is exercised here with two gloo ranks on the CPU, and the reference
arm's non-zero ranks exit without work."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    seconds = [0.5, 2.0][rank]
    slowest = bench.max_over_ranks(seconds)
    units = 1000 * (rank + 1)
    all_units = torch.tensor([units], dtype=torch.float64)
    dist.all_reduce(all_units)
    value = bench.aggregate([float(all_units.item())], [slowest])
    q.put((rank, slowest, value))
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 2.0                      # max over ranks
        assert abs(value - 3000 / 2.0) < 1e-9      # all units over the slowest rank


def test_max_over_ranks_without_group_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25) == 1.25


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_cpu_baseline_reports_all_cores_and_one_thread():
    """The oracle leg of the bench times the full decode on every host core
    and once on one thread; both figures are positive and the multi-thread
    result is the oracle's decode of the same inputs."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import oracle
    from paged_kv_continuous_gb300 import synth
    w = synth.tiny_decode()
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.store_kv(w.new_k, w.new_v, kc, vc, w.slot_mapping)
    ref, cpu = bench.cpu_baseline_oracle(w, kc, vc, seconds=0.05)
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["cores"] >= 1
    assert cpu["single_thread"]["cores"] == 1 and cpu["single_thread"]["value"] > 0
    assert np.array_equal(ref, oracle.decode(w.q, kc, vc, w.block_tables, w.context_lens,
                                             w.scale))
