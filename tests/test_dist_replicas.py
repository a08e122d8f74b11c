"""The N > 1 path of bench.py on the CPU: two gloo ranks (world size 2, 127.0.0.1).

The layer has no collective (replicas only), so the multi-process logic is bench.py's own: the
process-group set-up, the barrier around the timed region, the maximum of the step time over
ranks, the whole-job (weak-scaling) throughput, and rank 0 alone running the reference arm.
"""
import importlib.util
import os
import socket
import sys
import types

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    b = _bench()
    r, w, local = b.dist_init()
    assert (r, w, local) == (rank, ws, rank)
    b.barrier(ws)
    step_ms = 1.0 + 2.0 * rank  # ranks time different step lengths
    ms_max = b.max_over_ranks(step_ms, ws, "cpu")
    value = b.aggregate_tokens_per_s(4096, ws, ms_max)
    # the reference arm: only rank 0 does work; the others return at once without output
    ran = None
    if rank != 0:
        import io
        import contextlib
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            ran = b.reference_arm(types.SimpleNamespace(workload="tiny", steps=1, warmup=0, gpus=ws), rank, ws)
        assert ran is None and buf.getvalue() == ""
    b.barrier(ws)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{ms_max} {value}\n")
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.timeout(240)
def test_two_gloo_ranks(tmp_path):
    ws = 2
    mp.spawn(_rank_main, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, join=True)
    lines = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(ws)]
    for ms_max, value in lines:
        assert float(ms_max) == 3.0  # the slowest rank's step
        assert float(value) == pytest.approx(4096 * ws / 3.0e-3)


def test_single_process_is_the_identity():
    b = _bench()
    assert b.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert b.aggregate_tokens_per_s(4096, 1, 2.0) == pytest.approx(4096 / 2.0e-3)
