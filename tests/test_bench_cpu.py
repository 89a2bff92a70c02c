"""The bench's reference arm (the fp64 oracle on the host cores) prints one
JSON line with the contract's keys; it needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        # each rank timed a different span; every rank must see the slowest
        t = bench.reduce_max_over_ranks(1.5 + rank, world, "cpu")
        q.put((rank, t, bench.whole_job_rate(100, world, t)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_bench_takes_the_slowest_rank_with_two_gloo_ranks():
    """The N > 1 timing path on CPU: two gloo ranks reduce their timed spans to
    the maximum, and the whole-job rate divides all ranks' units by it."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gloo_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    assert [r[1] for r in res] == [2.5, 2.5]
    assert [r[2] for r in res] == [200 / 2.5, 200 / 2.5]


def test_reference_arm_under_two_ranks_prints_once():
    """Launched like the driver's N = 2 run, only rank 0 runs the oracle and
    prints; the other rank exits 0 without work."""
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """A committed ncu summary's DRAM bytes are reported only while its
    source_sha1 matches the kernel source; every kernel summary carries both
    lines and the command that made it."""
    import bench
    prof = os.path.join(bench.ROOT, "profiles")
    names = [f for f in os.listdir(prof) if f.endswith(".md") and not f.startswith("launches")]
    assert names
    for f in names:
        text = open(os.path.join(prof, f)).read()
        assert "ncu --set full --clock-control none" in text, f
        assert any(l.startswith("traffic_bytes_per_launch:") for l in text.splitlines()), f
        assert any(l.startswith("source_sha1:") for l in text.splitlines()), f
    # a summary whose hash matches is read; one whose hash does not is ignored
    sha = bench.kernel_source_hash()
    fake = tmp_path / "profiles"
    fake.mkdir()
    (fake / "k_w.md").write_text(f"x\ntraffic_bytes_per_launch: 1234\nsource_sha1: {sha}\n")
    (fake / "k_old.md").write_text("x\ntraffic_bytes_per_launch: 99\nsource_sha1: 000000000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: sha)
    assert bench.profiled_traffic("k", "w") == 1234.0
    assert bench.profiled_traffic("k", "old") is None
    assert bench.profiled_traffic("k", "missing") is None
