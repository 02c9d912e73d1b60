"""The replica path of bench.py on CPU: two gloo ranks, as torchrun would
start them, take distinct input seeds and agree on the slowest rank's time.
(The scan's rows are independent, so N GPUs run N replicas with no
collective on the data path; this is the only exchange.)"""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.rank_env()
    seed = bench.rank_seed("vim_s_1248_bimamba_v2", r)
    t = bench.max_over_ranks(1.0 + 2.0 * r, w)          # rank r "took" 1 + 2r ms
    dist.destroy_process_group()
    out.put((r, w, lr, seed, t))


def test_two_gloo_ranks_distinct_seeds_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, s0, t0), (r1, w1, l1, s1, t1) = res
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert s0 != s1 and s1 == s0 + 1
    assert t0 == t1 == 3.0


def test_single_rank_is_a_no_op(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.rank_env() == (1, 0, 0)
    assert bench.max_over_ranks(4.5, 1) == 4.5
