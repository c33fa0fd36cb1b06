"""The multi-GPU mode of the bench is replicas: every rank runs its own copy of
the workload and the job's time is the slowest rank's.  This checks the host
side of that aggregation with two gloo ranks on CPU (no GPU, no collective on
the data path)."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, tok = bench.aggregate_over_ranks(10.0 + 5.0 * rank, 1000 + rank)
    out[rank] = (ms, tok)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_timing_takes_the_slowest_rank_and_all_tokens():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        assert res[r] == (15.0, 2001.0)


def test_single_process_keeps_its_numbers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_over_ranks(3.5, 42) == (3.5, 42)


def test_every_package_name_the_bench_calls_is_exported():
    # the bench drives the library through the package namespace (gdn.<name>)
    import re
    import chunked_gated_delta_06_gb300 as gdn
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py")).read()
    names = set(re.findall(r"\bgdn\.([A-Za-z_]\w*)", src))
    assert names and not [n for n in sorted(names) if not hasattr(gdn, n)]
