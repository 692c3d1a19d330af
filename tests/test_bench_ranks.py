"""The benchmark's multi-rank path on CPU: two gloo ranks (replicas, no data-path collective).

Rank times differ; the job rate must use the slowest rank's time and every rank's units, and the
reference arm must print exactly one line, from rank 0, while rank 1 exits without work.
"""
import contextlib
import io
import json
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    import torch.distributed as dist
    bench.dist_setup("gloo")
    try:
        # rank r took (r + 1) * 100 ms for 50 tokens
        rate, ms = bench.job_rate(50, (rank + 1) * 100.0)
        bench.barrier()
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            rc = bench.main(["--impl", "reference", "--workload", "qwen3_layer_4bit",
                             "--layers", "1", "--steps", "1", "--warmup", "3"])
        q.put((rank, rate, ms, rc, buf.getvalue()))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_gloo_ranks_rate_and_reference_line():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, rate, ms, rc, out = q.get(timeout=300)
        got[rank] = (rate, ms, rc, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        rate, ms, rc, _ = got[rank]
        assert ms == pytest.approx(200.0)           # the slower rank's time
        assert rate == pytest.approx(2 * 50 / 0.2)  # both ranks' tokens
        assert rc == 0
    lines = [json.loads(l) for l in got[0][3].splitlines() if l.strip()]
    assert len(lines) == 1 and lines[0]["impl"] == "reference"
    assert lines[0]["cpu_baseline"]["kind"] == "oracle"
    assert lines[0]["e2e"]["h2d_bytes_per_step"] == 0
    assert got[1][3].strip() == ""
