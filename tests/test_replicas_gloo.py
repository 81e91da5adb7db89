"""The multi-GPU path of bench.py on CPU: two gloo ranks stand in for two replicas. Each rank
times its own layer; the job time is the slowest rank's, throughput counts every rank's tokens,
and the reference arm runs on rank 0 only."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r "measured" (2 + r) ms for the timed loop and (5 - r) ms end to end
        ms, ms_e2e = bench.max_over_ranks([2.0 + rank, 5.0 - rank], dist, "cpu")
        tput = bench.job_tokens_per_s(256, world, ms)
        # the reference arm: only rank 0 runs the oracle and prints its line
        args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0",
                                 "--config", "tiny", "--gpus", str(world)])
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(args, bench_cfg(), rank)
        printed = buf.getvalue()
        out[rank] = (ms, ms_e2e, tput, printed)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def bench_cfg():
    import synth
    return synth.get_config("tiny")


@pytest.mark.timeout(240)
def test_two_replicas_take_the_slowest_rank_and_count_every_rank():
    world = 2
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    for r in range(world):
        ms, ms_e2e, tput, _ = res[r]
        assert ms == 3.0 and ms_e2e == 5.0           # element-wise max over the two ranks
        assert tput == pytest.approx(2 * 256 / 3e-3)  # both ranks' tokens in the slowest time
    line = json.loads(res[0][3].strip())
    assert line["impl"] == "reference" and line["n_gpus"] == world and line["value"] > 0
    assert res[1][3] == ""                            # the other rank does no work
