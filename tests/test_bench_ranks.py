"""The multi-rank parts of bench.py without a GPU: two gloo ranks on CPU.
The layer forward has no exchange step, so N GPUs run N replicas; the bench
only needs the job time as the maximum over ranks, whole-job tokens/s from
it, and the reference arm on rank 0 alone."""
import importlib.util
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        # rank r took 10*(r+1) ms: the job took the slowest rank's time
        ms = b.max_over_ranks(10.0 * (rank + 1))
        value = b.job_value(100, 4, world, ms)

        class Args:
            gpus, steps, warmup = world, 1, 0
        buf = io.StringIO()
        with redirect_stdout(buf):
            rc = b.reference_arm(Args(), b.CONFIGS["toy"])
        out.put((rank, ms, value, rc, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    res = sorted(out.get() for _ in range(2))
    for rank, ms, value, rc, text in res:
        assert ms == 20.0                       # max over ranks, on every rank
        assert value == pytest.approx(2 * 100 * 4 / 0.020)
        assert rc == 0
    assert '"impl": "reference"' in res[0][4]   # rank 0 prints the reference line
    assert res[1][4] == ""                      # the other rank exits without work


def test_single_process_is_identity():
    b = _bench()
    assert not dist.is_initialized()
    assert b.max_over_ranks(3.5) == 3.5
    assert b.job_value(100, 2, 1, 1000.0) == 200.0
