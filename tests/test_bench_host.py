"""bench.py's multi-rank plumbing on the CPU: two gloo ranks agree on the max
time, and the throughput counts every rank's query heads (weak scaling)."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    world, r, _ = bench.dist_setup()
    slowest = bench.dist_max(world, 10.0 * (r + 1), "cpu")
    bench.dist_barrier(world)
    q.put((r, world, slowest, bench.throughput(world, 512, 100, slowest)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[0] for r in res] == [0, 1]
    for _, world, slowest, value in res:
        assert world == 2 and slowest == 20.0
        # 2 ranks x 512 query heads x 100 steps in 20 ms
        assert abs(value - 2 * 512 * 100 / 0.020) < 1e-6


def test_single_process_throughput():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.throughput(1, 512, 2000, 640.0) == 512 * 2000 / 0.64


def test_cpu_oracle_pool_matches_direct_calls():
    """The CPU baseline's process pool (spawn workers reading each (sequence, KV
    head) pair from shared memory) returns what the oracle returns when called
    directly, and reports the worker count as its cores."""
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    from long_context_sparse_score_gb300 import workloads as W
    from oracle import hashattn_oracle as O
    w = W.make_gqa(5, B=2, Hq=8, Hkv=2, d=64, n_cap=2048, seq_lens=[2048, 1500], m=100, n_sink=8,
                   n_local=16, device="cpu")
    secs, done, res, cores = bench.run_cpu_oracle(w, 12)
    assert done == 12 and len(res) == 12 and secs > 0
    assert cores == len(os.sched_getaffinity(0))
    q = w.q.float().numpy().astype(np.float64)
    for (b, h), (idx, _, out, lse) in res.items():
        g = h // 4
        want = O.decode_head(q[b, h], int(w.q_sig[b, h]),
                             w.k_sig[b, g].numpy().astype(np.int64), w.K[b, g].float().numpy(),
                             w.V[b, g].float().numpy(), int(w.seq_lens[b]), w.m, w.n_sink, w.n_local)
        assert np.array_equal(idx, want[0]) and np.array_equal(out, want[2]) and lse == want[3], (b, h)
