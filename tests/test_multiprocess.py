"""The bench's multi-process path on the CPU: two gloo ranks run the process-group setup, the
barrier and the max-over-ranks reduction that ``bench.py --gpus N`` uses under torchrun (each
rank runs an independent replica; only the timing is reduced)."""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_setup(world)
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 * (r + 1), w)
    planned = None
    import split_kv_decode_flash_gb300 as dattn
    import workloads as W
    wl = W.paged_ragged_gqa("cpu", B=4, lo=16, hi=200, pool_pages=64)
    planned = dattn.dattn_plan(wl.problem, wl.kv_len, page_indptr=wl.page_indptr, num_sms=8).info["n_items"]
    q.put((r, w, slowest, planned, dist.get_backend()))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_the_slowest_time():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert all(o[2] == 20.0 for o in out)            # max over ranks reaches every rank
    assert out[0][3] == out[1][3]                    # each replica plans the same work
    assert all(o[4] == "gloo" for o in out)


if __name__ == "__main__":
    pytest.main([__file__, "-q"])
