"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks (no GPU). Replicas do not exchange
data; the only collectives are the barrier around the timed region and the max over ranks of the
measured time, and the reference arm prints on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench._dist() == (ws, rank, rank)
        bench._barrier(ws)
        t = bench._max_over_ranks(ws, 10.0 + rank)   # rank 1 is the slow one
        out.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]


@pytest.mark.parametrize("config", ["stack80", "prefill80_t8", "gdn80", "gqa80_8k"])
def test_reference_arm_prints_on_rank_zero_only(capsys, monkeypatch, config):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.argparse.Namespace(config=config, steps=1, warmup=0, gpus=2, layers=0, ref_layers=1,
                                    ref_budget=0.1, no_cpu_baseline=True, impl="reference")
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
