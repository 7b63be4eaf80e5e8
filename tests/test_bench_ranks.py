"""Multi-rank logic of bench.py on CPU: two gloo ranks (no GPU)."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench = _bench()
    # each rank timed 10*(rank+1) ms for 100 samples: max time, summed samples
    out[rank] = bench.aggregate_over_ranks(10.0 * (rank + 1), 100, None)
    dist.destroy_process_group()


def test_timing_is_the_max_and_units_the_sum_over_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
        assert out[0] == (20.0, 200.0)
        assert out[1] == (20.0, 200.0)


def test_single_process_keeps_local_values():
    assert _bench().aggregate_over_ranks(3.5, 7, None) == (3.5, 7.0)


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    bench = _bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    bench.main()
    assert capsys.readouterr().out == ""
