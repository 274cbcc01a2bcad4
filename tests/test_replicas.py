"""The multi-GPU path of bench.py is replicas only: each rank prefills its
own prompt, with no collective on the data path; the ranks meet at a barrier
around the timed region and the job's time is the slowest rank's. This runs
that rank logic as two gloo processes on the CPU (no GPU, no prefill)."""
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench

    try:
        w, r, local, pg = bench.dist_setup()
        assert (w, r, local) == (world, rank, rank) and pg is not None
        bench.barrier(pg)
        ms = [12.5, 20.0][rank]  # this rank's own timed region
        slowest = bench.max_over_ranks(pg, ms)
        value = bench.replica_tok_per_s(w, 4096, 5, slowest / 1000.0)
        # the reference arm runs on rank 0 only: the other ranks return at once, without work
        ref_rc = bench.run_reference(None, None, w, r, pg) if r != 0 else None
        bench.barrier(pg)
        q.put((rank, slowest, value, ref_rc))
    finally:
        import torch.distributed as dist

        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_time_the_job_by_the_slowest_rank():
    torch = pytest.importorskip("torch")
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    # the children see no GPU, so the group is gloo on the CPU wherever this runs
    saved = os.environ.get("CUDA_VISIBLE_DEVICES")
    os.environ["CUDA_VISIBLE_DEVICES"] = ""
    try:
        for p in procs:
            p.start()
    finally:
        if saved is None:
            os.environ.pop("CUDA_VISIBLE_DEVICES", None)
        else:
            os.environ["CUDA_VISIBLE_DEVICES"] = saved
    try:
        res = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert [r[1] for r in res] == [20.0, 20.0]  # both ranks see the slowest rank's time
    assert res[0][2] == res[1][2] == 2 * 4096 * 5 / 0.020  # whole-job tokens over the job's time
    assert res[1][3] == 0  # rank 1's reference arm did nothing


def test_single_process_has_no_group():
    import bench

    env = {k: os.environ.pop(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.dist_setup() == (1, 0, 0, None)
        assert bench.max_over_ranks(None, 3.5) == 3.5
        assert bench.replica_tok_per_s(1, 4096, 2, 0.5) == 4096 * 2 / 0.5
    finally:
        os.environ.update(env)
