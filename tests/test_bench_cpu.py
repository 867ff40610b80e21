"""Host-side logic of bench.py without a GPU: clock-sample parsing, the traffic
record, the device-error report, the oracle CPU baseline on the tiny workload,
and the cross-rank aggregation with two gloo ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_clock_summary_keeps_samples_inside_the_timed_window():
    c = bench.ClockSampler(0)
    c.lines = [
        "2026/12/02 08:00:00.000, 0, 1980, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 08:00:01.000, 0, 1440, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 08:00:01.500, 0, 1500, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 08:00:03.000, 0, 2070, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    import datetime
    t = lambda s: datetime.datetime.strptime(s, "%Y/%m/%d %H:%M:%S.%f").timestamp()
    c.t0, c.t1 = t("2026/12/02 08:00:00.900"), t("2026/12/02 08:00:02.000")
    s = c.summary()
    assert s["samples_in_timed_region"] == 2 and s["sm_mhz"] == 1470.0
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070.0
    c.lines = ["garbage"]
    assert c.summary() is None


def test_recorded_traffic_requires_matching_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_digest", lambda: "abc123")
    (tmp_path / "profiles" / "decode_7b_traffic.md").write_text(
        "traffic_bytes_per_launch: 2.5e9\nsource_digest: abc123\npartition_size: 4096\n")
    assert bench.recorded_traffic("7b", 4096) == 2.5e9
    assert bench.recorded_traffic("7b", 512) is None            # taken at another partition size
    monkeypatch.setattr(bench, "source_digest", lambda: "changed")
    assert bench.recorded_traffic("7b", 4096) is None
    assert bench.recorded_traffic("8b", 4096) is None


def test_device_errors_are_named_with_their_bits():
    class FakeLib:
        DEVERR_BLOCK_ID, DEVERR_SLOT, DEVERR_CONTEXT, DEVERR_TIMEOUT, DEVERR_PREFIX = 1, 2, 4, 8, 16

        def __init__(self, bits):
            self.bits = bits

        def read_device_errors(self, dev_err, stream=None):
            return self.bits

    class Step:
        dev_err = None

    bench.check_device_errors(FakeLib(0), Step(), None, "warm-up")   # a clear word passes
    with pytest.raises(AssertionError, match=r"0x9 \(block id, timeout\) during the timed steps"):
        bench.check_device_errors(FakeLib(9), Step(), None, "the timed steps")


def test_host_inputs_pack_every_input_into_one_buffer(monkeypatch):
    import torch
    from paged_kv_cache_168_gb300.workloads import make_workload
    monkeypatch.setattr(torch.Tensor, "pin_memory", lambda self: self)   # no GPU here: pageable stands in
    w = make_workload("tiny", device="cpu")
    names = ("q", "key", "value", "block_tables", "context_lens", "slot_mapping")
    h = bench.HostInputs(w, names, "cpu")
    h.dev.fill_(0xAB)
    h.upload()                                    # one copy brings every input
    for k in names:
        a, b = getattr(w, k), h.views[k]
        assert a.dtype == b.dtype and a.shape == b.shape and torch.equal(a, b), k
        assert (b.data_ptr() - h.dev.data_ptr()) % 256 == 0
    assert h.nbytes == sum(-(-getattr(w, k).numel() * getattr(w, k).element_size() // 256) * 256 for k in names)
    # the prefill step's inputs (query_start_loc among them) travel the same way
    from paged_kv_cache_168_gb300.workloads import make_prefill_workload
    pw = make_prefill_workload("prefill_8b", device="cpu")
    pnames = ("q", "key", "value", "block_tables", "context_lens", "query_start_loc", "slot_mapping")
    ph = bench.HostInputs(pw, pnames, "cpu")
    ph.upload()
    for k in pnames:
        assert torch.equal(getattr(pw, k), ph.views[k]), k


def test_oracle_baseline_on_tiny_workload():
    from paged_kv_cache_168_gb300.workloads import make_workload
    w = make_workload("tiny")
    gbs, sps, desc, cores, secs = bench.oracle_sample(w, 0.05)
    assert gbs > 0 and sps > 0 and cores >= 1 and "tiny" in desc
    gbs1, _, desc1, cores1, _ = bench.oracle_sample(w, 0.05, threads=1)
    assert gbs1 > 0 and cores1 == 1 and "1 OpenMP threads" in desc1


def _rank(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        out[rank] = bench.reduce_max(10.0 + rank, world, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_over_ranks_with_gloo():
    with socket.socket() as sck:
        sck.bind(("127.0.0.1", 0))
        port = sck.getsockname()[1]
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 11.0, 1: 11.0}


def test_dist_env_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.reduce_max(3.5, 1, None) == 3.5
