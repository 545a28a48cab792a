"""The bench's multi-rank host logic on CPU: two gloo ranks (no GPU).

Covers what a torchrun launch of bench.py relies on besides the kernels:
the job time is the max over ranks, whole-job throughput counts every rank's
shard, each rank draws its own shard (rank 0's is the single-GPU workload),
and the reference arm does its work on rank 0 only.
"""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sinkhorn_mixing_gb300 import inputs  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    from sinkhorn_mixing_gb300 import inputs as inp
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        # per-rank step times: rank 1 is the slow one
        t = b.max_over_ranks([0.25, 0.75][rank], world, "cpu")
        wl = inp.WORKLOADS["tiny"]
        s = b.shard_streams(wl, 8, rank, "cpu")
        x = s["x"].view(torch.int16).to(torch.int64)
        sig = torch.tensor([float(x.sum()), float((x * x).sum())], dtype=torch.float64)
        sigs = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sigs, sig)
        dist.barrier()
        with open(os.path.join(outdir, "rank%d.json" % rank), "w") as f:
            json.dump({"t": t, "sigs": [v.tolist() for v in sigs],
                       "value": b.job_tokens_per_s(world, 8, 10, t)}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_max_and_distinct_shards(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    for r in res:
        assert r["t"] == 0.75                      # the slowest rank's time, on every rank
        assert r["value"] == pytest.approx(2 * 8 * 10 / 0.75)
    sigs = res[0]["sigs"]
    assert sigs == res[1]["sigs"]                  # both ranks saw the same gather
    assert sigs[0] != sigs[1]                      # the shards differ
    wl = inputs.WORKLOADS["tiny"]
    x0 = inputs.make_streams(wl, n=8, device="cpu")["x"].view(torch.int16).to(torch.int64)
    assert sigs[0] == [float(x0.sum()), float((x0 * x0).sum())]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.5, 1, "cpu") == 1.5
    assert bench.job_tokens_per_s(1, 65536, 500, 0.8) == pytest.approx(65536 * 500 / 0.8)


def test_shard_zero_is_the_single_gpu_workload():
    wl = inputs.WORKLOADS["tiny"]
    a = bench.shard_streams(wl, 8, 0, "cpu")["x"]
    b = inputs.make_streams(wl, n=8, device="cpu")["x"]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = bench.parse(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"])
    bench.run_reference(args, inputs.WORKLOADS["tiny"], rank=1)
    assert capsys.readouterr().out == ""


def test_traffic_record_only_for_its_workload_and_source(tmp_path, monkeypatch):
    # the committed DRAM traffic belongs to the large hc=4 workload and to the
    # kernel source it was captured on; any other workload or an edited
    # source reports no traffic
    import hashlib
    import json
    committed = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for kernel in ("hc_mixes_pre", "hc_post"):
        c = committed[kernel]
        current = hashlib.sha256(open(os.path.join(ROOT, c["source"]), "rb").read()).hexdigest()[:16]
        rec = bench.traffic_record(kernel, 4, 5120, 65536)
        assert (rec is not None) == (current == c["source_sha256_16"])
        if rec is not None:
            assert rec["dram_bytes_per_launch"] > 0
    assert bench.traffic_record("hc_post", 8, 5120, 65536) is None
    assert bench.traffic_record("hc_mixes_pre", 4, 5120, 16384) is None
    assert bench.traffic_record("hc_mixes_pre", 4, 2048, 65536) is None
    src = tmp_path / "k.cu"
    src.write_text("a")
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"hc_post": dict(
        committed["hc_post"], source="k.cu")}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("hc_post", 4, 5120, 65536) is None
    # the same record with the source's own hash is reported
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"hc_post": dict(
        committed["hc_post"], source="k.cu",
        source_sha256_16=hashlib.sha256(b"a").hexdigest()[:16])}))
    rec = bench.traffic_record("hc_post", 4, 5120, 65536)
    assert rec is not None and rec["dram_bytes_per_launch"] > 0
