"""Host-side logic of bench.py without a GPU: the multi-rank reduction of the
timed region (two gloo ranks on the CPU), the workload selection and the
recorded-traffic lookup keyed by the kernel's source hash."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed 1 + r seconds over 10 * (r + 1) work units
        seconds, units = bench.reduce_time_and_units(1.0 + rank, 10.0 * (rank + 1), world)
        results[rank] = (seconds, units)
    finally:
        dist.destroy_process_group()


def test_reduction_over_two_gloo_ranks():
    """The job's time is the slowest rank's, its work the sum of all ranks'."""
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        got = dict(results)
    assert got[0] == got[1] == (2.0, 30.0)


def test_single_rank_reduction_is_identity():
    assert bench.reduce_time_and_units(1.5, 7.0, 1) == (1.5, 7.0)


def test_workload_selection_and_head_override():
    args = bench.parse_args(["--workload", "video", "--heads", "24"])
    cfg = bench.select_workload(args)
    assert (cfg.B, cfg.H, cfg.S, cfg.D) == (1, 24, 17550, 64)
    assert bench.select_workload(bench.parse_args([])).H == 48
    with pytest.raises(SystemExit):
        bench.select_workload(bench.parse_args(["--heads", "0"]))


def test_recorded_traffic_needs_matching_source_hash(tmp_path, monkeypatch):
    profiles = tmp_path / "profiles"
    profiles.mkdir()
    h = bench.kernel_source_hash()
    (profiles / "traffic.txt").write_text(f"# header\nattn_fwd video {h} 123\nattn_fwd video deadbeef 456\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the source files are looked up under ROOT as well: point them at the real tree
    monkeypatch.setattr(bench, "kernel_source_hash", lambda names=bench.ATTN_SOURCES: h)
    assert bench.recorded_traffic("attn_fwd", "video") == 123.0
    assert bench.recorded_traffic("attn_fwd", "pixart_1024") is None
