"""Multi-rank host logic of the benchmark on CPU (gloo, world_size 2).

The path shards by rows: each rank runs its own replica and the ranks only
exchange scalars (max of timings, sum of bytes).  These tests run the
benchmark's reduction helpers in two gloo processes on 127.0.0.1."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, lr = bench.dist_init()
    assert (r, w, lr) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    mx = bench.reduce_scalar(1.5 + rank, "max")
    sm = bench.reduce_scalar(10.0 * (rank + 1), "sum")
    bench.barrier()
    q.put((rank, mx, sm))
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
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
    # max over ranks of the per-rank time, sum over ranks of the per-rank bytes
    assert got == [(0, 2.5, 30.0), (1, 2.5, 30.0)]


def test_single_rank_is_identity(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_init() == (0, 1, 0)
    assert bench.reduce_scalar(3.25, "max") == 3.25
    bench.barrier()


def test_bench_decode_bytes_match_the_recipe():
    """Algorithmic bytes of one decode call at B=256: state read + write
    (1 GiB), bf16 vectors, int32 counts, captured slots of rows with count >= 1."""
    sys.path.insert(0, ROOT)
    import bench
    counts = [0] * 56 + [1] * 50 + [2] * 50 + [3] * 50 + [4] * 50
    got = bench.decode_bytes(counts)
    state = 2 * 256 * 32 * 128 * 128 * 4
    vecs = 256 * (2 * 16 * 128 + 2 * 32 * 128 + 2 * 32) * 2 + 256 * 4
    slot = (32 + 16 * 128 + 32 * 128) * 4
    assert got == state + vecs + 200 * slot
    b, f = bench.prefill_bytes_flops()
    assert f == 4100 * 32 * (6 * 128 * 128 + 10 * 64 * 128)


def test_bench_verify_bytes_match_the_recipe():
    """Algorithmic bytes of one fused replay + verify call at B=256, state in
    place: the state read for every row and written for rows that replay,
    replayed slots read, 4 draft tokens' bf16 inputs and outputs, 4 captured
    slots written per row, int32 counts."""
    sys.path.insert(0, ROOT)
    import bench
    accepted = [0] * 56 + [1] * 50 + [2] * 50 + [3] * 50 + [4] * 50
    got = bench.verify_bytes(accepted, 256)
    st = 32 * 128 * 128 * 4
    slot = (32 + 16 * 128 + 32 * 128) * 4
    tokens = 256 * 4 * (2 * 16 * 128 + 2 * 32 * 128 + 2 * 32) * 2
    replayed = 50 * (1 + 2 + 3 + 4)
    assert got == 256 * st + 200 * st + replayed * slot + 256 * 4 * slot + 2 * 256 * 4 + tokens
