"""The multi-process path of the benchmark (N independent replicas), run as
two gloo ranks on the CPU: the slowest rank's times win, the whole-job rate
counts every rank's units, and a single process is left alone."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

from exact_attention_94_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        own = [10.0 + rank, 5.0 * (rank + 1), 3.0 - rank]  # ranks disagree in both directions
        slowest = replicas.max_over_ranks(own)
        replicas.barrier()
        rate = replicas.whole_job_rate(world, 100.0, slowest[0])
        e2e = replicas.rescale_to_slowest(50.0, own[0], slowest[0], world)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "rate": rate, "e2e": e2e}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["slowest"] == [11.0, 10.0, 3.0]           # element-wise max over the ranks
        assert r["rate"] == pytest.approx(2 * 100.0 / 0.011)  # both ranks' units at the slowest time
    assert res[0]["e2e"] == pytest.approx(2 * 50.0 * 10.0 / 11.0)
    assert res[1]["e2e"] == pytest.approx(2 * 50.0 * 11.0 / 11.0)


def test_single_process_is_untouched():
    assert replicas.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert replicas.whole_job_rate(1, 10.0, 2.0) == pytest.approx(5000.0)
    with pytest.raises(ValueError):
        replicas.whole_job_rate(0, 1.0, 1.0)
