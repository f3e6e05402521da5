"""Host logic of bench.py without a GPU: the multi-rank aggregation (max over
ranks, whole-job throughput) on two gloo ranks, clock parsing, and the JSON
contract of the reference arm (run whole, on one rank and under a two-rank
torchrun: it times the oracle on the host and needs no GPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    local_seconds = [0.50, 0.80][rank]          # rank 1 is the slowest
    m = bench.reduce_max(local_seconds, world)
    bench.barrier(world)
    agg = bench.aggregate(1e12, 10, world, m)
    q.put((rank, m, agg))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, agg in res:
        assert m == 0.80
        # 2 ranks x 10 steps x 1e12 flops over the slowest rank's 0.8 s
        assert agg["value"] == pytest.approx(2 * 10 * 1e12 / 0.8 / 1e12)
        assert agg["ms_per_step"] == pytest.approx(80.0)


def test_single_rank_is_identity():
    assert bench.reduce_max(1.25, 1) == 1.25
    assert bench.aggregate(2e12, 4, 1, 2.0)["value"] == pytest.approx(4.0)


def test_clock_sampler_parsing():
    s = bench.ClockSampler(0)
    s.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout=None: 0})()
    s.lines = ["0, 1965, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    r = s.stop()
    assert r["sm_mhz"] == pytest.approx((1965 + 2070) / 2)
    assert r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]
    assert r["samples"] == 2


def test_traffic_requires_matching_kernel_hash(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "shared_memory_operand_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    h = bench.kernel_source_hash()
    (prof / f"{bench.KERNEL_NAME}_w.md").write_text(
        f"kernel_source_hash: {h}\ndram_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic("w") == 123456.0
    assert bench.profiled_bank_conflicts("w") is None        # no shared-memory counters in this summary
    (csrc / "k.cu").write_text("kernel v2")
    assert bench.profiled_traffic("w") is None


def test_bank_conflicts_from_profile(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "shared_memory_operand_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    h = bench.kernel_source_hash()
    (prof / f"{bench.KERNEL_NAME}_w.md").write_text(
        f"# title\n\nkernel_source_hash: {h}\ndram_bytes_per_launch: 1e6\nsmem_st_requests: 1000\n"
        "smem_st_bank_conflicts: 50\nsmem_ld_requests: 10\nsmem_ld_bank_conflicts: 0\n"
        "smem_excess_wavefronts: 0\nl2_to_sm_bytes_per_launch: 4096\n\n| table | 12 |\n")
    c = bench.profiled_bank_conflicts("w")
    assert c["st_per_request"] == pytest.approx(0.05)
    assert c["ld_per_request"] == 0.0
    assert c["excess_wavefronts"] == 0 and c["st_requests"] == 1000
    assert bench.profiled_traffic("w") == 1e6
    assert bench.profiled_counters("w")["l2_to_sm_bytes_per_launch"] == 4096
    (csrc / "k.cu").write_text("kernel v2")
    assert bench.profiled_bank_conflicts("w") is None


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_single_rank():
    """`bench.py --impl reference` times the oracle on the host (no GPU needed)
    and prints one JSON line carrying the contract's keys."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--workload", "gemm_256_bf16_f32"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["metric"] == "BF16 GEMM TFLOP/s" and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_two_ranks_prints_once():
    """Under torchrun with two ranks only rank 0 runs and prints; both exit 0."""
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port),
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "3",
                        "--warmup", "3", "--workload", "gemm_256_bf16_f32"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference"
