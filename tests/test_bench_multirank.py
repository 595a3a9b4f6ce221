"""Host logic of bench.py's multi-rank path (independent replicas under
torch.distributed), run with world sizes 2 and 4 over gloo on the CPU: every
rank gets the slowest rank's time, the whole-job value counts every rank's work
over that time, and the reference arm prints from rank 0 only."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        out[rank] = bench.max_over_ranks(1.5 + 2.0 * rank, world, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        slowest = 1.5 + 2.0 * (world - 1)
        assert dict(out) == {r: slowest for r in range(world)}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, 1, "cpu") == 4.25


def test_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_gbs(10**9, 1, 1.0) == pytest.approx(1000.0)
    assert bench.job_gbs(10**9, 4, 2.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_0_only():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        workload, steps, warmup, ref_requests = "c0", 1, 0, 1
    assert bench.run_reference(A(), 1, 2) is None


def test_pages_baseline_only_for_the_pages_own_shapes():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.pages_baseline_gbs("c1q4") == pytest.approx(730.0)
    assert bench.pages_baseline_gbs("p-16-150000") == pytest.approx(1700.0)
    assert bench.pages_baseline_gbs("c1q1") is None
    assert bench.pages_baseline_gbs("c3") is None


@pytest.mark.parametrize("name,kind", [
    ("c0", "dense"), ("c1q1", "dense"), ("c1q4", "dense"), ("c2-2x4096", "dense"),
    ("c4-1", "sparse"), ("c4x-1", "sparse"), ("d-2-16-3-100", "dense"),
    ("p-2-256", "dense"), ("dcp2-c0", "dcp"),
])
def test_every_workload_name_parses(name, kind):
    sys.path.insert(0, ROOT)
    import bench
    k, inp, desc = bench.make_workload(name)
    assert k == kind and desc
    assert bench.kv_bytes_per_call(k, inp) == bench.keys_per_call(k, inp) * bench.row_bytes(k)


def test_packed_buffers_are_256_byte_aligned_views():
    sys.path.insert(0, ROOT)
    import bench
    import torch
    ts = [torch.arange(5, dtype=torch.int32), torch.ones(3, 7, dtype=torch.bfloat16),
          torch.zeros(1, dtype=torch.float32)]
    buf, views = bench._packed(ts)
    for v, t in zip(views, ts):
        assert v.shape == t.shape and v.dtype == t.dtype
        assert (v.data_ptr() - buf.data_ptr()) % 256 == 0
        v.copy_(t)
    for v, t in zip(views, ts):
        assert torch.equal(v, t)


def _gloo_max(argv):
    # a spawn_ranks target: the rank's environment is set as torchrun sets it
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo")
    try:
        rank, world = dist.get_rank(), dist.get_world_size()
        assert int(os.environ["LOCAL_RANK"]) == rank and world == int(os.environ["WORLD_SIZE"])
        got = bench.max_over_ranks(10.0 + rank, world, "cpu")
        with open(os.path.join(argv[0], f"rank{rank}"), "w") as f:
            f.write(f"{world} {got}")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_spawn_ranks_runs_one_process_per_rank_with_torchrun_env(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    bench.spawn_ranks(2, [str(tmp_path)], target=_gloo_max)
    assert sorted(os.listdir(tmp_path)) == ["rank0", "rank1"]
    for r in (0, 1):
        assert open(tmp_path / f"rank{r}").read() == "2 11.0"


def test_bench_gpus_2_spawns_ranks_and_prints_one_line():
    # `bench.py --gpus 2` without torchrun launches two ranks itself; the
    # reference arm runs on rank 0 only, so exactly one JSON line comes out
    import json
    import subprocess
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--impl", "reference", "--workload", "c0", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
    # the same workload label and sizes as the GPU arm's config
    sys.path.insert(0, ROOT)
    import bench
    kind, inp, desc = bench.make_workload("c0")
    assert out["config"]["workload"] == bench.workload_label("c0", kind, desc)
    assert out["config"]["kv_bytes_per_call"] == bench.kv_bytes_per_call(kind, inp)
    assert out["config"]["keys_per_call"] == bench.keys_per_call(kind, inp)


def test_every_sweep_workload_name_parses():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.ALL_WORKLOADS[1] == "c1q1"
    for name in bench.ALL_WORKLOADS:
        if name.startswith(("c2-", "c3")):
            continue   # large pools; the names share their parser with c2-2x4096 above
        k, inp, desc = bench.make_workload(name)
        assert desc
