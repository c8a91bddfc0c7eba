"""Host logic of bench.py: aggregation over ranks (gloo, world size 2, on
CPU), clock-record parsing, traffic records, and the reference arm's
behaviour on ranks other than 0."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_aggregate_is_all_ranks_tokens_over_max_time():
    r = bench.aggregate([10.0, 20.0], tokens_per_step=4096, steps=5)
    assert r["ms_per_step"] == 4.0
    assert r["value"] == pytest.approx(4096 * 5 * 2 / 0.020)


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    m = bench.reduce_max(10.0 * (rank + 1), dist, torch.device("cpu"))
    agg = bench.aggregate([m] * world, 100, 2)
    q.put((rank, m, agg["value"]))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [m for _, m, _ in res] == [20.0, 20.0]
    assert all(v == pytest.approx(100 * 2 * 2 / 0.020) for _, _, v in res)


def test_clock_summary_parsing():
    c = bench.ClockSampler("0")
    c.lines = ["0, 1900, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1800, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 1850, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active"]
    s = c.summary()
    assert s["sm_mhz"] == 1850 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]


def test_traffic_record_tied_to_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for rel in bench.SOURCE_FILES:
        p = tmp_path / rel
        p.parent.mkdir(parents=True, exist_ok=True)
        p.write_text("kernel source v1")
    (tmp_path / "profiles").mkdir()
    d = bench.source_digest()
    (tmp_path / "profiles" / "traffic.txt").write_text(
        f"# comment\nphase=fwd_lse_gemm workload=qwen source={d} dram_bytes_per_launch=123.5\n")
    assert bench.recorded_traffic("fwd_lse_gemm", "qwen") == 123.5
    assert bench.recorded_traffic("bwd_dE_gemm", "qwen") is None
    (tmp_path / bench.SOURCE_FILES[0]).write_text("kernel source v2")
    assert bench.recorded_traffic("fwd_lse_gemm", "qwen") is None


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0


def test_warmup_must_be_three_or_more():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_per_config_covers_every_workload_and_filter_mode():
    """The default run reports every workload and filter mode besides the
    headline, plus the single call and the all-rows forward on the
    long-context batch."""
    import cce_workloads as W
    cases = bench.per_config_cases("long", "on", False, True)
    want = {(n, f) for n in W.CONFIG_ORDER for f in W.CONFIGS[n].filter_modes} - {("long", "on")}
    assert {(n, f) for n, f, sgl, skp in cases if not sgl and skp} == want
    assert ("long", "on", True, True) in cases
    assert ("long", "on", False, False) in cases
    assert len(cases) == len(want) + 2
