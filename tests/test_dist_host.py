"""Replica aggregation across ranks (host logic of bench.py's N>1 path),
run as two gloo ranks on CPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, nbytes = bench.aggregate_over_ranks(10.0 + 5.0 * rank, 1000 * (rank + 1), world, backend_device="cpu")
        results[rank] = (ms, nbytes)
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        for r in range(2):
            ms, nbytes = results[r]
            assert ms == 15.0          # the slowest rank's time
            assert nbytes == 3000.0    # the work of all ranks


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate_over_ranks(3.5, 42, 1) == (3.5, 42)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("M", [1, 32])
def test_bench_bytes_match_oracle_count(M):
    import bench
    import oracle
    for fmt, od in bench.FORMATS:
        assert bench.algorithmic_bytes(M, fmt, od) == oracle.algorithmic_bytes(M, 16, fmt, od)
    for fmt, _ in bench.V_FORMATS:
        assert bench.v_up_algorithmic_bytes(M, fmt) == oracle.v_up_algorithmic_bytes(M, 16, fmt)


def test_committed_traffic_table_is_consistent():
    # The roofline's `traffic` comes from the committed ncu table while the
    # kernel sources still hash to the value recorded in it.  When they do,
    # the table must cover every (pair, M) the bench times, and each launch's
    # DRAM bytes must sit near the algorithmic reads (weights, scales and q;
    # the output stays in L2 within the launch).
    import bench
    table = bench.measured_traffic()
    if table is None:
        pytest.skip("the kernel sources changed since the committed ncu capture")
    for fmt, od in bench.FORMATS:
        key = f"{fmt}->{od}"
        for M in bench.M_POINTS:
            assert (key, M) in table, (key, M)
            out_bytes = M * 16 * 576 * (2 if od == "bf16" else 1)
            reads = bench.algorithmic_bytes(M, fmt, od) - out_bytes
            assert 0.98 * reads <= table[(key, M)] <= 1.05 * reads, (key, M, table[(key, M)], reads)
