"""The benchmark's host-side logic on CPU: the multi-rank (replicas) path with
world size 2 over gloo -- each rank runs an independent replica, the job's time
is the slowest rank's and the throughput counts the units of every rank -- and
the roofline's traffic figure taken from a committed ncu summary."""
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = 1.0 + rank                      # rank 1 is slower
        bench.barrier(world)
        t_max = bench.max_over_ranks(t, world)
        out[rank] = (t_max, bench.job_throughput(100, world, t_max))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, 2, 29511, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1] == (2.0, 100.0)   # 2 ranks x 100 units / 2 s


@pytest.mark.slow
def test_reference_arm_two_ranks_prints_one_line():
    """Under torchrun with two ranks only rank 0 times the oracle and prints."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", "29512", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--L", "512"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1 and '"impl": "reference"' in lines[0]


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """The headline roofline's DRAM traffic comes from the committed ncu summary
    only while the kernel source still hashes to what was profiled."""
    import hashlib
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    # the committed summary against the committed source
    t = bench.profiled_traffic("scan_sd_tc_diag_B8x2048_H32.md", "linear_attention_state_gated_gb300/csrc/scan_sd_tc.cu")
    assert t is not None and t > 2e9
    # a copy of the tree whose kernel source differs: no traffic figure
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k").mkdir()
    src = tmp_path / "k" / "kernel.cu"
    src.write_text("// kernel v1\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "s.md").write_text(
        "# summary\n| metric | value |\ntraffic_bytes_per_launch_L8192: 1234\nsource_sha256_prefix: " + sha + "\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("s.md", "k/kernel.cu") == 1234.0
    src.write_text("// kernel v2\n")
    assert bench.profiled_traffic("s.md", "k/kernel.cu") is None
    assert bench.profiled_traffic("missing.md", "k/kernel.cu") is None
