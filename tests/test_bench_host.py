"""Host-side logic of bench.py that needs no GPU: the max-over-ranks
aggregation across processes (gloo, world size 2), the derived ALU peak, the
JSON line of the reference arm (the fp64 oracle on the host cores)."""

import io
import json
import os
import socket
from contextlib import redirect_stdout

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    mx = bench.aggregate_max(10.0 * (rank + 1), world)
    bench.barrier(world)
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(repr(mx))
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [float(open(tmp_path / f"r{r}.txt").read()) for r in range(2)]
    assert got == [20.0, 20.0]


def test_single_rank_aggregate_is_identity():
    import bench

    assert bench.aggregate_max(3.5, 1) == 3.5


def test_alu_peak_formula():
    import bench

    # 152 SMs x 128 fp32 lanes x 2070 MHz, 5 instructions per double-float MAC, 2 flops per MAC
    assert abs(bench.alu_peak_tflops(2070.0) - 152 * 128 * 2070e6 * 2 / 5 / 1e12) < 1e-9


def test_reference_arm_json_line():
    import bench

    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--config", "c1", "--steps", "2", "--warmup", "1", "--ref-rows", "32"])
    assert rc == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "weights/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["config"]["workload"] == "c1_64x64_Z"


def test_clock_sampler_without_nvidia_smi(monkeypatch):
    import bench

    def boom(*a, **k):
        raise OSError("no nvidia-smi")

    monkeypatch.setattr(bench.subprocess, "Popen", boom)
    c = bench.ClockSampler(0)
    c.start()
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_profiled_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    import shutil

    import bench

    for rel in bench.KERNEL_SOURCES:
        os.makedirs(tmp_path / os.path.dirname(rel), exist_ok=True)
        shutil.copy(os.path.join(ROOT, rel), tmp_path / rel)
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("chunk_push", "c3") is None  # no summary
    digest = bench.kernel_source_digest()
    (tmp_path / "profiles" / "chunk_push_c3_dram.json").write_text(
        json.dumps({"traffic_bytes_per_launch": 123456, "source_sha256": digest}))
    assert bench.profiled_traffic("chunk_push", "c3") == 123456
    with open(tmp_path / bench.KERNEL_SOURCES[0], "a") as f:
        f.write("\n// a comment edited\n/* and\n another */\n")
    assert bench.profiled_traffic("chunk_push", "c3") == 123456  # comments do not change the code
    with open(tmp_path / bench.KERNEL_SOURCES[0], "a") as f:
        f.write("\nstatic int edited = 1;\n")
    assert bench.profiled_traffic("chunk_push", "c3") is None  # stale once the code changes


def test_roofline_tensor_and_alu_classes():
    import bench

    peaks = {"bf16_tflops": 2000.0, "sm_max_mhz": 2000.0}
    r = bench.roofline_for("chunk_push", 1e12, 100.0, peaks)  # 10 TFLOP/s of fp64-equivalent products
    assert r["bound"] == "tensor" and abs(r["achieved"] - 200.0) < 1e-9 and abs(r["frac"] - 0.1) < 1e-12
    assert abs(r["alg_tflops_fp64_equiv"] - 10.0) < 1e-12 and r["peak_basis"].startswith("measured")
    assert bench.roofline_for("chunk_push", 1e12, 100.0, {})["peak_basis"].startswith("fallback")
    a = bench.roofline_for("tile_solve", 1e12, 100.0, peaks)
    assert a["bound"] == "alu" and abs(a["peak"] - bench.alu_peak_tflops(2000.0)) < 1e-12


def test_antidiagonal_work_count_by_brute_force():
    """Algorithm 3's multiply-adds with triangular factors: entry (p, q)
    receives one per earlier entry (i, j), i <= p, j <= q."""
    import bench

    for m, n in [(1, 1), (2, 3), (5, 4), (7, 9)]:
        brute = sum(1 for p in range(m) for q in range(n) for i in range(p + 1) for j in range(q + 1)
                    if (i, j) != (p, q))
        assert bench.antidiag_macs(m, n) == brute


def test_pages_same_shape_context():
    import bench

    c = bench.pages_same_shape(4096, 4096, 16.0)
    assert c["seconds"] == 0.288 and abs(c["ratio_pages_over_this"] - 18.0) < 1e-9
    assert bench.pages_same_shape(64, 64, 0.1) is None
