"""Host-side multi-process logic of the benchmark on CPU (gloo, world size 2).

Every rank moves its own replica; the whole-job throughput is the bytes of
all ranks divided by the slowest rank's time.  No GPU is involved here.
"""
import io
import json
import os
import socket
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    d = bench.init_dist(world, "gloo")
    seconds = [0.5, 2.0][rank]
    units = [100.0, 300.0][rank]
    bench.barrier(d)
    total_units, max_seconds = bench.aggregate(d, seconds, units)
    out.put((rank, total_units, max_seconds))
    dist.destroy_process_group()


def test_aggregate_takes_slowest_rank_and_sums_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=10) for _ in range(2))
    for rank, units, seconds in results:
        assert units == 400.0 and seconds == 2.0


def test_single_process_aggregate_is_identity():
    import bench

    assert bench.aggregate(None, 1.5, 42.0) == (42.0, 1.5)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert buf.getvalue() == ""


def test_reference_arm_prints_contract_line(monkeypatch):
    import bench

    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-tiles", "16"])
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_bench_rejects_short_warmup():
    import bench

    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_traffic_is_reported_only_for_the_kernel_it_was_measured_on(monkeypatch, tmp_path):
    import hashlib

    import bench

    src = tmp_path / "kernel.cu"
    src.write_text("// kernel source\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    profile = tmp_path / "profile.md"
    profile.write_text(f"    traffic_bytes_per_launch: 1234567\n    kernel_source_sha256_16: {digest}\n")
    monkeypatch.setattr(bench, "KERNEL_SOURCES", [str(src)])
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(profile))
    assert bench.committed_traffic()[0] == 1234567
    src.write_text("// kernel source, changed\n")
    value, why = bench.committed_traffic()
    assert value is None and "changed" in why
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(tmp_path / "missing.md"))
    assert bench.committed_traffic()[0] is None


def test_in_bound_bytes_of_workload4_agree_with_the_oracle_fill_mask():
    # the algorithmic bytes of the workload-4 lines: every box byte the engine
    # reads rather than fills, counted two independent ways
    import numpy as np

    import bench
    import datagen
    import oracle

    w = datagen.C4
    coords = datagen.workload_coords(w)
    v = oracle.View(w.esize, w.dims, w.strides, w.box, w.swizzle)
    filled = int(oracle.tile_oob_mask(v, coords).astype(np.int64).sum())
    inb = bench.box_inbound_bytes(w.dims, w.box, w.esize, coords)
    assert inb == len(coords) * oracle.box_bytes(v) - filled
    assert inb == 29_045_120  # the figure the workload-4 profiles quote
