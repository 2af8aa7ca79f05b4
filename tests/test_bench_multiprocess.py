"""bench.py's multi-process host logic on CPU: gloo, world size 2.

Covers the max-over-ranks timing and whole-job aggregation the bench uses
under torchrun, and the reference arm's rank handling (rank 0 alone runs and
prints; the other ranks exit 0 without work).
"""

import json
import os
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 0.010 + 0.005 * rank  # rank 1 is the slow replica
        slowest = bench.max_over_ranks(local, dist, torch.device("cpu"))
        q.put((rank, slowest, bench.aggregate_value(0.002, slowest, world)))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_max_over_ranks_and_aggregate_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert abs(slowest - 0.015) < 1e-12  # every rank sees the slowest replica's time
        assert abs(value - 100.0 * 0.002 / 0.015 * 2) < 1e-9


def test_single_process_helpers_without_a_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, None, None) == 0.5
    assert abs(bench.aggregate_value(1.0, 2.0, 1) - 50.0) < 1e-12


def test_roofline_is_rated_against_the_burst_peak():
    """Tensor-bound kernels are rated against the burst bf16 figure whatever the clock record says;
    when the power cap held the median clock down, the fraction of the sustained figure is added as a
    note. HBM-bound kernels are always rated against the copy figure."""
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0, "source": "measured"}
    burst = bench.roofline_entry("k", "tensor", 1.6e12, 1e-3, peaks, None)
    assert burst["peak"] == 2000.0 and abs(burst["frac"] - 0.8) < 1e-9
    assert abs(burst["frac_of_burst"] - 0.8) < 1e-9 and "frac_of_sustained" not in burst
    capped_clk = {"sm_mhz": 1400.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    capped = bench.roofline_entry("k", "tensor", 1.6e12, 1e-3, peaks, 123, capped_clk)
    assert capped["peak"] == 2000.0 and abs(capped["frac"] - 0.8) < 1e-9 and capped["traffic"] == 123
    assert abs(capped["frac_of_sustained"] - 1.0) < 1e-9 and "note" in capped
    # the cap flagged but the clock at its maximum: no sustained note
    full_clk = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert "frac_of_sustained" not in bench.roofline_entry("k", "tensor", 1.6e12, 1e-3, peaks, None, full_clk)
    hbm = bench.roofline_entry("k", "hbm", 3e9, 1e-3, peaks, None, capped_clk)
    assert hbm["peak"] == 6000.0 and abs(hbm["frac"] - 0.5) < 1e-9 and "frac_of_burst" not in hbm


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed table while the kernel source still has the hash it was
    captured at; a changed source, a missing source or an unknown key gives null."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel v1")
    digest = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# header line\n"
        f"w:0 k.cu {digest} 12345\n"
        "w:1 missing.cu 0000000000000000 7\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("w:0") == 12345
    assert bench.load_traffic("w:1") is None
    assert bench.load_traffic("w:2") is None
    src.write_bytes(b"kernel v2")
    assert bench.load_traffic("w:0") is None


def test_committed_traffic_table_names_existing_sources():
    """Every row of the committed table names a kernel source of this repository and a 16-hex digest."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert rows
    for key, src, digest, byts in rows:
        assert ":" in key and os.path.exists(os.path.join(ROOT, src)), (key, src)
        assert len(digest) == 16 and int(digest, 16) >= 0 and int(byts) > 0


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "2", "--warmup", "1", "--reference-seconds", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
