"""Host logic of the benchmark's multi-rank path on CPU: two gloo ranks, the max-over-ranks
time, the whole-job throughput, and the reference arm's rank-0-only rule.  Each rank of a
real run processes its own full batch (weak scaling); nothing on the data path crosses
ranks, so these are the only cross-rank steps."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    t = bench.reduce_max(0.5 + rank, w)          # rank 1 is the slow one
    v = bench.aggregate(800, w, t)
    dist.barrier()
    dist.destroy_process_group()
    out.put((r, w, local, t, v))


def _run_two_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(out.get(timeout=120) for _ in procs)
    except Exception:
        res = None
    for p in procs:
        p.join(timeout=60)
        if p.exitcode is None:
            p.kill()
    ok = res is not None and all(p.exitcode == 0 for p in procs)
    return res if ok else None


def test_two_gloo_ranks_take_the_max_time_and_sum_the_work():
    # the free port can be taken by another process between the probe and the rendezvous:
    # a second attempt gets a new one
    res = _run_two_ranks() or _run_two_ranks()
    assert res is not None, "two gloo ranks did not complete"
    for rank, (r, w, local, t, v) in enumerate(res):
        assert (r, w, local) == (rank, 2, rank)
        assert t == 1.5                    # max over ranks
        assert v == pytest.approx(800 * 2 / 1.5)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    assert bench.aggregate(10, 1, 2.0) == 5.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_its_line(monkeypatch, capsys):
    import json
    sys.path.insert(0, ROOT)
    import bench
    for var in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3", "--workload", "c1_tiny"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "queries/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_gpus_n_without_torchrun_spawns_n_ranks_for_the_reference_arm():
    # the reference arm under N self-spawned ranks: rank 0 alone prints its line
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3", "--workload", "c1_tiny"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_gpus_n_without_enough_gpus_is_an_error():
    import subprocess

    import torch
    if torch.cuda.device_count() >= 64:
        pytest.skip("a machine with 64 GPUs")
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "64", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode != 0 and "visible GPUs" in r.stderr
    assert not any(x.startswith("{") for x in r.stdout.splitlines())


def test_spawn_command_runs_torchrun_on_localhost():
    sys.path.insert(0, ROOT)
    import bench
    cmd = bench.spawn_command(4, ["--steps", "5"], 12345)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert cmd[cmd.index("--nproc-per-node") + 1] == "4"
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-2:] == ["--steps", "5"]


def test_rotation_count_keeps_three_l2_between_uses():
    sys.path.insert(0, ROOT)
    import bench

    class FakeStep:
        def __init__(self, hbm):
            self.hbm = hbm

        def bytes(self):
            return {"hbm": self.hbm}

    l2 = 126 << 20
    for hbm in (84 << 20, 571 << 20, 10 << 20, 3 << 30):
        n = bench.rotation_count(FakeStep(hbm), l2)
        assert n >= 2
        assert (n - 1) * hbm >= 3 * l2          # enough other traffic between two uses of a copy
        assert n == 2 or (n - 2) * hbm < 3 * l2  # and no more copies than that needs


def test_cluster_step_takes_block_selection_over_short_rows():
    sys.path.insert(0, ROOT)
    import bench
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS
    assert bench.cluster_step_supported(WORKLOADS["c3_block_sparse"])
    for name in ("c1_tiny", "c2_llama3_8b_gqa", "c4_tiered_verify", "c6_window_blocks", "c7_head_topk"):
        assert not bench.cluster_step_supported(WORKLOADS[name])
    w = WORKLOADS["c3_block_sparse"]
    assert not bench.cluster_step_supported(w.scaled(block=48))   # runs must be whole 16/32-row pieces
    assert not bench.cluster_step_supported(w.scaled(T=64 * 8196))  # more blocks than one cluster holds


def test_tiered_attention_oracle_step_leaves_t3_out():
    # the CPU reference of the tiered step at a small size: with every position in T0 it is the
    # plain dense attention; with the tiers it differs (T2 quantised, T3 gone)
    import math

    import numpy as np

    import oracle
    sys.path.insert(0, ROOT)
    import bench
    from top_sparse_decode_gqa_gb300.workloads import WORKLOADS, generate
    w = WORKLOADS["c11_tiered_attention"].scaled(T=1024, layers=2, Hq=8, Hkv=2)
    x = generate(w)
    res = bench.oracle_step(w, x, 0, 1)
    assert len(res) == w.layers
    plain = oracle.gather_attend(x["q"][0, 0, 0:1].contiguous(), x["k"][0][0:1].contiguous(),
                                 x["v"][0][0:1].contiguous(), None, 1, w.V, w.Hq, w.Hkv, w.d, w.T, w.T, 1,
                                 1 / math.sqrt(w.d))[0]
    out, lse = res[0]
    assert out.shape == plain.shape and np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    assert not np.allclose(out, plain, atol=1e-6)
