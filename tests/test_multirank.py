"""The N > 1 plumbing of bench.py on CPU: two gloo ranks (127.0.0.1).

bench.py runs one independent replica per GPU ("replicas only": output rows
shard with no collective, and every rank streams its own weight buffers); the
only cross-rank steps are the barriers around the timed region, the maximum
of the ranks' times, and the reference arm printing from rank 0 alone."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, local = bench.dist_init(backend="gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    t = bench.allmax(w, 0.25 * (rank + 1))          # rank r "took" 0.25 (r + 1) s
    # the reference arm: rank 0 prints its one JSON line, the others return at once
    class A:
        ref_rows, steps, warmup, gpus = 64, 1, 1, world
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A())
    bench.barrier(w)
    dist.destroy_process_group()
    out.put((rank, t, buf.getvalue()))


@pytest.mark.timeout(300)
def test_two_gloo_ranks_agree_on_the_slowest_time_and_rank0_reports():
    pytest.importorskip("torch")
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        rank, t, printed = q.get(timeout=240)
        res[rank] = (t, printed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 0.5              # both ranks see the slowest rank's time
    import json
    line = json.loads(res[0][1].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert res[1][1] == ""                              # rank 1 prints nothing
