"""Host logic of bench.py: the roofline model the pages use, clock-sample
parsing, and max-over-ranks aggregation across world_size-2 gloo ranks."""
import os
import socket

import pytest

import bench


def test_roofline_worked_numbers():
    # Section "A rough way to ask how much room was left": the pooler's 64 MiB
    # of weights at 4.8e12 B/s is about 13.98 µs; 2·16·4096·8192 FLOPs at
    # 989e12 FLOP/s about 1.09 µs; M = 256 makes the FLOP bound about 17.37 µs.
    wbytes = 2 * 4096 * 8192
    assert wbytes == 64 * 2**20
    t = bench.roofline_time_s(wbytes, 0, 4.8e12, 989e12)
    assert round(t * 1e6, 2) == 13.98
    assert round(bench.roofline_time_s(0, 2 * 16 * 4096 * 8192, 4.8e12, 989e12) * 1e6, 2) == 1.09
    assert round(bench.roofline_time_s(0, 2 * 256 * 4096 * 8192, 4.8e12, 989e12) * 1e6, 2) == 17.37
    # The bound is the slower of the two (bytes at M = 16).
    assert bench.roofline_time_s(wbytes, 2 * 16 * 4096 * 8192, 4.8e12, 989e12) == t
    # Weight-only arithmetic intensity is M FLOPs per weight byte.
    for M in (1, 16, 256):
        assert 2 * M * 4096 * 8192 / wbytes == M


def test_clock_summary():
    rows = [["0", "2070", "2070", "700.5", "0x0", "Not Active", "Not Active", "Not Active",
             "Not Active"],
            ["0", "1900", "2070", "1300.0", "0x4", "Not Active", "Not Active", "Not Active",
             "Active"],
            ["0", "1950", "2070", "1200.0", "0x4", "Not Active", "Not Active", "Not Active",
             "Active"]]
    c = bench.summarize_clocks(rows)
    assert c["sm_mhz"] == 1950 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3


def test_profile_traffic_requires_matching_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILE_DIR", str(tmp_path))
    (tmp_path / "proj_tc_kernel_x.md").write_text(
        "traffic_bytes_per_launch: 123\nkernel_source_sha256: deadbeef\n")
    assert bench.profile_traffic("x")[0] is None
    (tmp_path / "proj_tc_kernel_x.md").write_text(
        f"traffic_bytes_per_launch: 123\nkernel_source_sha256: {bench.kernel_source_hash()}\n")
    assert bench.profile_traffic("x")[0] == 123


def test_args_contract():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.impl == "gb300" and a.workload == "decode_bias"
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # Rank r processed 10 units in r+1 seconds: the job's time is the slowest
    # rank's, its throughput all units over that time.
    agg = bench.aggregate_throughput(10.0, float(rank + 1))
    out[rank] = (agg["seconds"], agg["units"], agg["per_second"])
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == (2.0, 20.0, 10.0)


def test_reference_arm_is_rank0_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference_arm(bench.parse_args(["--impl", "reference"])) is None
